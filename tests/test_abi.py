"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/diffattn.h declares, and rejects bad arguments on the host
before any CUDA call."""
import ctypes
import os
import re

import pytest

import differential_attention_diffattn_gb300 as da
from differential_attention_diffattn_gb300 import _lib
from oracle import oracle as orc

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "diffattn.h")


@pytest.fixture(scope="module")
def lib():
    da.build()
    return da.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \t\*]*?\b(diffattn_[a-z0-9_]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTED), names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_lambda_init_host(lib):
    for depth in (1, 2, 8, 12, 24, 100):
        assert abs(da.diffattn_lambda_init(depth) - orc.lambda_init(depth)) < 1e-7
    assert da.diffattn_lambda_init(0) != da.diffattn_lambda_init(0)  # NaN


def test_status_strings(lib):
    for s in range(7):
        assert da.diffattn_status_string(s) != "unknown status"
    assert da.diffattn_status_string(99) == "unknown status"


FAKE = 0x10000  # aligned, never dereferenced: every case below fails validation first


def _desc(**kw):
    d = _lib.DiffAttnDesc()
    base = dict(batch=1, seqlen=16, num_heads=4, num_kv_heads=2, d=64, dv=128, dtype=_lib.DTYPE_BF16, eps=1e-5)
    base.update(kw)
    for k, v in base.items():
        setattr(d, k, v)
    return d


def _fwd(lib, desc, q=FAKE, k=FAKE, v=FAKE, lam=FAKE, w=FAKE, out=FAKE, cu=None):
    vp = ctypes.c_void_p
    return lib.diffattn_fwd(ctypes.byref(desc), vp(q), vp(k), vp(v), vp(lam), 0, 0.2, vp(w), 1,
                            vp(cu) if cu else None, vp(out), None)


@pytest.mark.parametrize("kw,ptrs,want", [
    (dict(num_heads=3), {}, 1),                 # H % Hkv != 0
    (dict(dv=64), {}, 1),                       # dv != 2d
    (dict(num_heads=0), {}, 1),
    (dict(batch=-1), {}, 1),
    (dict(eps=-1.0), {}, 1),
    (dict(dtype=7), {}, 1),
    ({}, dict(q=0), 1),                         # null pointer
    ({}, dict(out=0), 1),
    ({}, dict(q=FAKE + 8), 1),                  # not 16-byte aligned
    (dict(d=32, dv=64), {}, 2),                 # bf16 only with d = 64
    (dict(d=128, dv=256, dtype=_lib.DTYPE_F32), {}, 2),
    (dict(batch=0), {}, 0),                     # empty: nothing to launch
])
def test_fwd_rejects_on_host(lib, kw, ptrs, want):
    assert _fwd(lib, _desc(**kw), **ptrs) == want


def test_forward_kernel_choice(lib):
    # items of at most 64 key tiles, at least two per SM, at most 64 packed
    # sequences: the persistent kernel (the library assumes 152 SMs when no GPU
    # answers; a GB300 has 152)
    def kernel(packed=0, **kw):
        name = lib.diffattn_fwd_kernel(ctypes.byref(_desc(**kw)), packed)
        return name.decode() if name else None
    assert kernel(batch=4, seqlen=2048, num_heads=16, num_kv_heads=4) == "diffattn_fwd_bf16_persistent_kernel"
    assert kernel(batch=3, seqlen=1000, num_heads=16, num_kv_heads=4) == "diffattn_fwd_bf16_persistent_kernel"
    assert kernel(batch=1, seqlen=16384, num_heads=16, num_kv_heads=16) == "diffattn_fwd_bf16_sm103a_kernel"
    assert kernel(batch=2, seqlen=512, num_heads=16, num_kv_heads=4) == "diffattn_fwd_bf16_sm103a_kernel"
    assert kernel(packed=1, num_seqs=14, max_seqlen=4096, total_tokens=32768, num_heads=16,
                  num_kv_heads=4) == "diffattn_fwd_bf16_persistent_kernel"
    assert kernel(packed=1, num_seqs=65, max_seqlen=4096, total_tokens=65536, num_heads=16,
                  num_kv_heads=4) == "diffattn_fwd_bf16_sm103a_kernel"
    assert kernel(packed=1, num_seqs=2, max_seqlen=256, total_tokens=356, num_heads=16,
                  num_kv_heads=4) == "diffattn_fwd_bf16_sm103a_kernel"
    assert kernel(batch=2, seqlen=8192, num_heads=16, num_kv_heads=4) == "diffattn_fwd_bf16_persistent_kernel"
    assert kernel(batch=1, seqlen=8193, num_heads=16, num_kv_heads=4) == "diffattn_fwd_bf16_sm103a_kernel"
    assert kernel(batch=1, seqlen=32768, num_heads=16, num_kv_heads=16) == "diffattn_fwd_bf16_sm103a_kernel"
    assert kernel(d=16, dv=32, dtype=_lib.DTYPE_F32) == "diffattn_fwd_f32_kernel"
    assert kernel(d=32, dv=64) is None


def test_varlen_argument_checks(lib):
    d = _desc(num_seqs=-1, max_seqlen=16, total_tokens=16)
    assert _fwd(lib, d, cu=FAKE) == 1
    d = _desc(num_seqs=2, max_seqlen=16, total_tokens=16)
    assert _fwd(lib, d, cu=FAKE + 2) == 1       # misaligned cu_seqlens
    d = _desc(num_seqs=0, max_seqlen=0, total_tokens=0)
    assert _fwd(lib, d, cu=FAKE) == 0


def test_lambda_rejects_on_host(lib):
    vp = ctypes.c_void_p
    assert lib.diffattn_lambda(vp(FAKE), vp(FAKE), vp(FAKE), None, 1, 16, 0.2, vp(FAKE), None) == 1
    assert lib.diffattn_lambda(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 0, 16, 0.2, vp(FAKE), None) == 1
    assert lib.diffattn_lambda(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1, 0, 0.2, vp(FAKE), None) == 1


def test_binding_refuses_missing_library(tmp_path):
    with pytest.raises(RuntimeError):
        _lib.load_library(str(tmp_path / "missing.so"))


def _rope_desc(**kw):
    d = _lib.DiffAttnRopeDesc()
    base = dict(tokens=16, num_heads=4, num_kv_heads=2, d=64, dtype=_lib.DTYPE_BF16, rot_dim=64, interleaved=1,
                n_pos=16, num_seqs=0, seqlen=16)
    base.update(kw)
    for k, v in base.items():
        setattr(d, k, v)
    return d


def _rope(lib, desc, pos=None, cu=None, cos=FAKE, sin=FAKE, q=FAKE, qo=FAKE, k=FAKE, ko=FAKE):
    vp = ctypes.c_void_p
    w = lambda x: vp(x) if x else None  # noqa: E731
    return lib.diffattn_rope_qk(ctypes.byref(desc), w(pos), w(cu), w(cos), w(sin), w(q), w(qo), w(k), w(ko), None)


@pytest.mark.parametrize("kw,ptrs,want", [
    (dict(rot_dim=32), {}, 1),                  # neither d nor 2d
    (dict(d=12, rot_dim=12), {}, 1),            # rot_dim % 8 != 0
    (dict(n_pos=0), {}, 1),
    (dict(dtype=5), {}, 1),
    (dict(seqlen=0), {}, 1),                    # no position source
    (dict(num_seqs=0), dict(cu=FAKE), 1),       # cu_seqlens without sequences
    ({}, dict(q=0), 1),
    ({}, dict(k=0), 1),                         # k missing while num_kv_heads > 0
    ({}, dict(cos=FAKE + 4), 1),                # misaligned table
    ({}, dict(pos=FAKE + 2), 1),                # misaligned positions
    (dict(tokens=0), {}, 0),                    # empty: nothing to launch
])
def test_rope_rejects_on_host(lib, kw, ptrs, want):
    assert _rope(lib, _rope_desc(**kw), **ptrs) == want


def test_rope_tables_reject_on_host(lib):
    vp = ctypes.c_void_p
    assert lib.diffattn_rope_tables(10000.0, 0, 64, vp(FAKE), vp(FAKE), None) == 1
    assert lib.diffattn_rope_tables(10000.0, 8, 63, vp(FAKE), vp(FAKE), None) == 1
    assert lib.diffattn_rope_tables(-1.0, 8, 64, vp(FAKE), vp(FAKE), None) == 1
    assert lib.diffattn_rope_tables(10000.0, 8, 64, None, vp(FAKE), None) == 1


def test_cache_forward_split_plan(lib):
    # The library-planned split count of the cache forward, seen through the
    # workspace it needs: B q_len H splits (m, l, O of both components) in fp32.
    # The plan takes the fewest waves of resident split CTAs (2 per SM; the
    # library assumes 152 SMs when no GPU answers) whose last wave is at least
    # 80 % full: 8 sequences x 4 kv heads -> 9 splits (288 CTAs of 304 slots);
    # 16 x 4 -> 4 splits (256 of 304); a forced count is taken as given.
    def ws(batch, q_len, cap, H=16, Hkv=4, splits=0):
        d = _lib.DiffAttnKvDesc(batch=batch, q_len=q_len, cache_capacity=cap, num_heads=H, num_kv_heads=Hkv,
                                d=64, dv=128, dtype=_lib.DTYPE_BF16, eps=1e-5, num_splits=splits)
        return lib.diffattn_fwd_kvcache_workspace_size(ctypes.byref(d))
    per_split = lambda batch, q_len, H=16: batch * q_len * H * 2 * (128 + 2) * 4  # noqa: E731
    assert ws(8, 1, 16384) == 9 * per_split(8, 1)
    assert ws(16, 4, 8192) == 4 * per_split(16, 4)
    assert ws(16, 4, 8192, splits=7) == 7 * per_split(16, 4)
    assert ws(0, 1, 16384) == 0


def test_noalloc_cache_forward_checks_the_descriptor_first(lib):
    # A descriptor that diffattn_fwd_kvcache rejects as INVALID_ARG gets the same
    # status from the allocation-free entry, not a size rejection: a negative dv
    # would otherwise wrap the unsigned partials size to a huge number.
    vp = ctypes.c_void_p

    def call(**kw):
        base = dict(batch=4, q_len=1, cache_capacity=4096, num_heads=16, num_kv_heads=4, d=64, dv=128,
                    dtype=_lib.DTYPE_BF16, eps=1e-5, num_splits=0)
        base.update(kw)
        d = _lib.DiffAttnKvDesc(**base)
        return lib.diffattn_fwd_kvcache_noalloc(ctypes.byref(d), vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), 0,
                                                0.2, vp(FAKE), 1, vp(FAKE), None)
    assert call(dv=-128) == 1
    assert call(dv=-128, batch=1 << 20) == 1
    assert call(batch=70000) == 1       # above the batch limit
    assert call(num_heads=15) == 1      # heads not a multiple of kv heads
    assert call(d=32, dv=64) == 2       # valid, but no kernel for d = 32


def test_fault_injection_hook_is_off_without_the_test_environment(lib, monkeypatch):
    monkeypatch.delenv("DIFFATTN_TEST_HOOKS", raising=False)
    assert lib.diffattn_set_fault_injection(1) == 2   # UNSUPPORTED: left off
    assert lib.diffattn_set_fault_injection(0) == 2
    monkeypatch.setenv("DIFFATTN_TEST_HOOKS", "1")
    assert lib.diffattn_set_fault_injection(3) == 1   # no such mode
    assert lib.diffattn_set_fault_injection(1) == 0
    assert lib.diffattn_set_fault_injection(0) == 0


def test_cache_forward_split_plan_from_host_lengths(lib):
    # With a host copy of the lengths the plan models the split CTAs' streaming
    # time (fitted to GB300 sweeps; 152 SMs assumed without a GPU): the ragged
    # 16 x 4-token batch takes 7 splits (4 from the shape), the full 8 x 16k one 8.
    rag = [6638, 4932, 6735, 1706, 6830, 4356, 1178, 6860, 1195, 5839, 1610, 7005, 5464, 6260, 5740, 1016]

    def ws(batch, q_len, cap, lens):
        d = _lib.DiffAttnKvDesc(batch=batch, q_len=q_len, cache_capacity=cap, num_heads=16, num_kv_heads=4,
                                d=64, dv=128, dtype=_lib.DTYPE_BF16, eps=1e-5, num_splits=0)
        arr = (ctypes.c_int * batch)(*lens)
        d.host_seqlens = ctypes.cast(arr, ctypes.c_void_p)
        return lib.diffattn_fwd_kvcache_workspace_size(ctypes.byref(d))
    per_split = lambda batch, q_len: batch * q_len * 16 * 2 * (128 + 2) * 4  # noqa: E731
    assert ws(16, 4, 8192, rag) == 7 * per_split(16, 4)
    assert ws(8, 1, 16384, [16384] * 8) == 8 * per_split(8, 1)


def test_fwd_lambda_rejects_on_host(lib):
    """The combined lambda + forward call checks all its arguments before it
    launches anything (no GPU here: a launch would fail with ERR_CUDA)."""
    vp = ctypes.c_void_p

    def call(vecs=(FAKE, FAKE, FAKE, FAKE), lam_d=64, lam_out=FAKE, **desc_kw):
        base = dict(batch=1, seqlen=256, num_heads=16, num_kv_heads=4, d=64, dv=128, dtype=_lib.DTYPE_BF16, eps=1e-5)
        base.update(desc_kw)
        d = _lib.DiffAttnDesc(**base)
        return lib.diffattn_fwd_lambda(ctypes.byref(d), vp(FAKE), vp(FAKE), vp(FAKE), *(vp(x) for x in vecs), 0, lam_d,
                                       0.2, vp(lam_out), vp(FAKE), 1, None, vp(FAKE), None)
    assert call(vecs=(FAKE, 0, FAKE, FAKE)) == 1   # a null lambda vector
    assert call(lam_d=0) == 1
    assert call(lam_d=2000) == 1
    assert call(lam_out=0) == 1
    assert call(lam_out=FAKE + 2) == 1              # misaligned lambda output
    assert call(num_heads=15) == 1                  # the forward's own checks come first too
    assert call(d=32, dv=64) == 2                   # no bf16 kernel for d = 32
    assert call(batch=0) == 0                       # empty: nothing launched


def test_kvcache_lambda_rejects_on_host(lib):
    """The combined lambda + cache forward call checks all its arguments before it
    launches anything (no GPU here: a launch would fail with ERR_CUDA)."""
    vp = ctypes.c_void_p

    def call(vecs=(FAKE, FAKE, FAKE, FAKE), lam_d=64, lam_out=FAKE, ws_bytes=1 << 30, **desc_kw):
        base = dict(batch=4, q_len=1, cache_capacity=4096, num_heads=16, num_kv_heads=4, d=64, dv=128,
                    dtype=_lib.DTYPE_BF16, eps=1e-5, num_splits=0)
        base.update(desc_kw)
        d = _lib.DiffAttnKvDesc(**base)
        return lib.diffattn_fwd_kvcache_lambda(ctypes.byref(d), vp(FAKE), vp(FAKE), vp(FAKE), None,
                                               *(vp(x) for x in vecs), 0, lam_d, 0.2, vp(lam_out), vp(FAKE), 1,
                                               vp(FAKE), ws_bytes, vp(FAKE), None)
    assert call(vecs=(FAKE, FAKE, 0, FAKE)) == 1   # a null lambda vector
    assert call(lam_d=0) == 1
    assert call(lam_d=2000) == 1
    assert call(lam_out=0) == 1
    assert call(lam_out=FAKE + 2) == 1              # misaligned lambda output
    assert call(num_heads=15) == 1                  # the cache forward's own checks come first too
    assert call(ws_bytes=16) == 1                   # workspace too small
    assert call(d=32, dv=64) == 2                   # no kernel for d = 32
    assert call(batch=0) == 0                       # empty: nothing launched


def test_fused_rope_forward_rejects_on_host(lib):
    vp = ctypes.c_void_p

    def call(rope_kw=None, **desc_kw):
        base = dict(batch=1, seqlen=256, num_heads=16, num_kv_heads=4, d=64, dv=128, dtype=_lib.DTYPE_BF16, eps=1e-5)
        base.update(desc_kw)
        d = _lib.DiffAttnDesc(**base)
        rope = None
        if rope_kw is not None:
            r = dict(cos=FAKE, sin=FAKE, n_pos=1024, rot_dim=128, interleaved=0)
            r.update(rope_kw)
            rope = ctypes.byref(_lib.DiffAttnRopeQ(**r))
        return lib.diffattn_fwd_rope_q(ctypes.byref(d), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 0, 0.2, vp(FAKE),
                                       1, None, rope, vp(FAKE), None)
    assert call(None) == 1                           # no rotary tables
    assert call(dict(rot_dim=96)) == 1               # neither d nor 2d
    assert call(dict(rot_dim=12), d=12, dv=24) == 1  # not a multiple of 8
    assert call(dict(n_pos=0)) == 1
    assert call(dict(interleaved=2)) == 1
    assert call(dict(cos=FAKE + 4)) == 1             # misaligned table
    assert call(dict(sin=0)) == 1
    assert call(dict(), dtype=_lib.DTYPE_F32) == 2   # the fp32 path has no fused rotation
    assert call(dict(), batch=0) == 0                # empty: nothing launched


def test_rope_k_only_and_neither_on_host(lib):
    d = _rope_desc(num_heads=0, num_kv_heads=0)
    assert _rope(lib, d) == 1
