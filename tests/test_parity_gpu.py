"""GPU parity of the C-ABI path against the fp64 oracle (element by element).

Sizes the oracle finishes in seconds are compared in full; the two largest
workloads (T = 16384 and the 32k-token packed batch) are compared on sampled
rows, launched exactly as the benchmark launches them.
"""
import numpy as np
import pytest
import torch

import differential_attention_diffattn_gb300 as da
from differential_attention_diffattn_gb300 import workloads as W
from oracle import oracle as orc

from gpu_util import compare, oracle_out, row_condition, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    da.build()
    da.load_library()
    torch.cuda.set_device(0)


# -------------------------------------------------------------- lambda ---

@pytest.mark.parametrize("shape", [(16,), (64,), (16, 64), (3, 1000)])
def test_lambda_kernel(shape):
    g = torch.Generator().manual_seed(3)
    vs = [torch.randn(shape, generator=g) * 0.3 for _ in range(4)]
    li = da.diffattn_lambda_init(7)
    got = da.diffattn_lambda(*[x.cuda() for x in vs], li).cpu().numpy()
    want = orc.lambda_values(*vs, orc.lambda_init(7))
    np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-6)


def test_lambda_zero_vectors_give_lambda_init():
    z = torch.zeros(64, device="cuda")
    li = da.diffattn_lambda_init(12)
    got = da.diffattn_lambda(z, z, z, z, li).item()
    assert got == li


# ---------------------------------------------------------- workloads ---

@pytest.mark.parametrize("name", ["tiny_f32", "b2_t512_gqa", "llama1b_b4_t2048"])
def test_workload_full(name):
    inp = W.generate(W.WORKLOADS[name], seed=0)
    got = run_gpu(inp, packed=False)
    compare(got, oracle_out(inp), inp.wl.dtype)


@pytest.mark.parametrize("name", ["long_t16384", "varlen_32k"])
def test_workload_sampled(name):
    inp = W.generate(W.WORKLOADS[name], seed=0)
    got = run_gpu(inp, packed=name == "varlen_32k")
    assert torch.isfinite(got).all()
    tt, hh = sample_rows(inp)
    compare(got[torch.as_tensor(tt).long(), torch.as_tensor(hh).long()], oracle_out(inp, rows=(tt, hh)),
            inp.wl.dtype)


def test_bf16_long_sequence_65536():
    """The longest case: one 65536-token sequence (16 heads over 4 kv heads, 512
    query tiles, 268 MB per q / out tensor), compared on sampled rows."""
    inp = W.generate(W.with_overrides(W.WORKLOADS["b2_t512_gqa"], random_subln=True), seed=65, seq_lens=[65536])
    got = run_gpu(inp, packed=False)
    assert torch.isfinite(got).all()
    tt, hh = sample_rows(inp, every=997, edge=64)
    compare(got[torch.as_tensor(tt).long(), torch.as_tensor(hh).long()], oracle_out(inp, rows=(tt, hh)), "bf16")


# ---------------------------------------------------------- edge cases ---

BF = W.WORKLOADS["b2_t512_gqa"]


@pytest.mark.parametrize("T", [1, 2, 127, 128, 129, 255, 1000])
def test_bf16_ragged_lengths(T):
    inp = W.generate(BF, seed=T, seq_lens=[T])
    compare(run_gpu(inp), oracle_out(inp), "bf16")


@pytest.mark.parametrize("lens", [[1, 130, 7, 256, 3], [640, 1], [129, 129, 129], [4096, 33]])
def test_bf16_packed(lens):
    inp = W.generate(BF, seed=len(lens), seq_lens=lens)
    compare(run_gpu(inp), oracle_out(inp), "bf16")


def test_bf16_many_short_packed_sequences():
    # 2000 packed sequences of 1..48 tokens: the one-item-per-CTA kernel (more than
    # 64 packed sequences), with the sequences along the grid's slowest dimension.
    # This seed's lambda is 0.937, so among the 780k rows some nearly cancel
    # (kappa up to 24): each row's max-abs bound scales with its kappa
    lens = np.random.default_rng(17).integers(1, 49, 2000).tolist()
    inp = W.generate(BF, seed=17, seq_lens=lens)
    lam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2,
                            orc.lambda_init(inp.wl.depth))
    compare(run_gpu(inp), oracle_out(inp), "bf16", kappa=row_condition(inp, lam))


@pytest.mark.parametrize("T", [1, 100, 300])
def test_bf16_non_causal(T):
    inp = W.generate(W.with_overrides(BF, causal=False), seed=5, seq_lens=[T, 77])
    compare(run_gpu(inp), oracle_out(inp), "bf16")


@pytest.mark.parametrize("H,Hkv", [(16, 1), (16, 2), (16, 16), (3, 3), (8, 4)])
def test_bf16_head_groups(H, Hkv):
    inp = W.generate(W.with_overrides(BF, num_heads=H, num_kv_heads=Hkv), seed=H * 10 + Hkv, seq_lens=[300])
    compare(run_gpu(inp), oracle_out(inp), "bf16")


def test_bf16_per_head_lambda_and_random_weight():
    wl = W.with_overrides(BF, lambda_per_head=True, random_subln=True)
    inp = W.generate(wl, seed=11, seq_lens=[257, 190])
    compare(run_gpu(inp), oracle_out(inp), "bf16")


@pytest.mark.parametrize("lam", [0.0, 1.0, 1.9, -0.5])
def test_bf16_forced_lambda(lam):
    """lambda = 0 (plain attention), lambda = 1, lambda > 1, lambda < 0. Rows
    whose two maps nearly cancel are ill-conditioned, so the max-abs bound of
    each row scales with its kappa (see gpu_util.row_condition)."""
    inp = W.generate(BF, seed=21, seq_lens=[333])
    compare(run_gpu(inp, lam_value=lam), oracle_out(inp, lam_value=lam), "bf16",
            kappa=row_condition(inp, lam))


def test_bf16_large_scores():
    """Scores of a few hundred: exercises the deferred-rescale threshold."""
    inp = W.generate(BF, seed=22, seq_lens=[700])
    inp.q = (inp.q.float() * 6).to(torch.bfloat16)
    inp.k = (inp.k.float() * 6).to(torch.bfloat16)
    compare(run_gpu(inp), oracle_out(inp), "bf16")


# -------------------------------------- persistent kernel (unpacked) ---

@pytest.mark.parametrize("B,T,H,Hkv,causal,per_head", [(3, 1000, 16, 4, True, False), (5, 700, 12, 3, True, False),
                                                       (4, 2048, 16, 4, False, False), (12, 256, 16, 16, True, False),
                                                       (4, 1000, 16, 4, True, True), (64, 130, 16, 4, True, False)])
def test_bf16_persistent_kernel(B, T, H, Hkv, causal, per_head):
    """Unpacked batches with 2 to 10 (query tile, head, sequence) items per SM run
    on the persistent kernel: ragged last tiles, grouped kv heads, non-causal,
    many short items, a lambda per head."""
    wl = W.with_overrides(BF, num_heads=H, num_kv_heads=Hkv, causal=causal, random_subln=True,
                          lambda_per_head=per_head)
    inp = W.generate(wl, seed=B * 100 + T, seq_lens=[T] * B)
    sh = lambda x: x.cuda().view(B, T, *x.shape[1:])  # noqa: E731
    lam = torch.ones(1, dtype=torch.float32, device="cuda")
    assert da.diffattn_fwd_kernel(sh(inp.q), sh(inp.k), sh(inp.v), lam,
                                  inp.subln_w.cuda()) == "diffattn_fwd_bf16_persistent_kernel"
    compare(run_gpu(inp, packed=False), oracle_out(inp), "bf16")


def test_bf16_persistent_kernel_packed_large_scores():
    """Packed sequences on the persistent kernel with q and k scaled by 6 (scores of a
    few hundred): later tiles whose row sums pass 2^32 are taken maximum-first from
    scores recomputed on the CUDA cores, with keys at each sequence's own offset."""
    wl = W.with_overrides(BF, num_heads=16, num_kv_heads=4)
    lens = [700, 130, 1024, 257, 900, 64, 511, 1000, 384, 777]
    inp = W.generate(wl, seed=41, seq_lens=lens)
    inp.q = (inp.q.float() * 6).to(torch.bfloat16)
    inp.k = (inp.k.float() * 6).to(torch.bfloat16)
    t = inp.cu_seqlens.cuda()
    lam = torch.ones(1, dtype=torch.float32, device="cuda")
    assert da.diffattn_fwd_kernel(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), lam, inp.subln_w.cuda(), cu_seqlens=t,
                                  max_seqlen=max(lens)) == "diffattn_fwd_bf16_persistent_kernel"
    compare(run_gpu(inp), oracle_out(inp), "bf16")


def test_bf16_persistent_kernel_longest_items_sampled():
    """2 x 8192 tokens (items of up to 64 key tiles, the longest the persistent
    kernel takes), 16 / 4 heads, against the oracle on sampled rows."""
    B, T = 2, 8192
    wl = W.with_overrides(W.WORKLOADS["llama1b_b4_t2048"], random_subln=True)
    inp = W.generate(wl, seed=91, seq_lens=[T] * B)
    sh = lambda x: x.cuda().view(B, T, *x.shape[1:])  # noqa: E731
    lam = torch.ones(1, dtype=torch.float32, device="cuda")
    assert da.diffattn_fwd_kernel(sh(inp.q), sh(inp.k), sh(inp.v), lam,
                                  inp.subln_w.cuda()) == "diffattn_fwd_bf16_persistent_kernel"
    got = run_gpu(inp, packed=False)
    assert torch.isfinite(got.float()).all()
    tt, hh = sample_rows(inp, every=97)
    compare(got[torch.as_tensor(tt).long(), torch.as_tensor(hh).long()], oracle_out(inp, rows=(tt, hh)), "bf16")


@pytest.mark.parametrize("d,lens", [(16, [64, 3]), (32, [100]), (64, [70, 1])])
def test_f32_shapes(d, lens):
    wl = W.with_overrides(W.WORKLOADS["tiny_f32"], d=d, dv=2 * d, num_heads=4, num_kv_heads=2,
                          random_subln=True)
    inp = W.generate(wl, seed=d, seq_lens=lens)
    compare(run_gpu(inp), oracle_out(inp), "f32")


def test_f32_non_causal():
    wl = W.with_overrides(W.WORKLOADS["tiny_f32"], causal=False)
    inp = W.generate(wl, seed=4, seq_lens=[50, 13])
    compare(run_gpu(inp), oracle_out(inp), "f32")


# ------------------------------------------------------- equivalences ---

def test_batch_equals_separate_calls_bitwise():
    inp = W.generate(BF, seed=31, seq_lens=[300, 300, 300])
    full = run_gpu(inp, packed=False)
    for s in range(3):
        one = W.generate(BF, seed=31, seq_lens=[300, 300, 300])
        a, b = s * 300, (s + 1) * 300
        one.q, one.k, one.v = one.q[a:b], one.k[a:b], one.v[a:b]
        one.seq_lens, one.cu_seqlens = [300], torch.tensor([0, 300], dtype=torch.int32)
        assert torch.equal(run_gpu(one), full[a:b])


# 3 x 1000 tokens, 16 / 4 heads (8 key tiles an item); 3 x 8192 tokens, 2 heads
# (items of up to 64 key tiles, the longest the persistent kernel takes); q and k
# scaled by 6 (scores of a few hundred: rows whose maximum rises past the rescale
# threshold after the first tile, where the one-item-per-CTA kernel redoes the
# tile maximum-first)
@pytest.mark.parametrize("T,H,Hkv,qk_scale", [(1000, 16, 4, 1.0), (8192, 2, 2, 1.0), (1000, 16, 4, 6.0)])
def test_persistent_and_per_tile_kernels_agree_bitwise(T, H, Hkv, qk_scale):
    """An unpacked batch of three sequences runs on the persistent kernel, each
    sequence alone on the one-item-per-CTA kernel: the same bits."""
    wl = W.with_overrides(BF, num_heads=H, num_kv_heads=Hkv)

    def gen():
        g = W.generate(wl, seed=32, seq_lens=[T] * 3)
        if qk_scale != 1.0:
            g.q = (g.q.float() * qk_scale).to(torch.bfloat16)
            g.k = (g.k.float() * qk_scale).to(torch.bfloat16)
        return g

    inp = gen()
    B = 3
    sh = lambda x: x.cuda().view(B, T, *x.shape[1:])  # noqa: E731
    lam = torch.ones(1, dtype=torch.float32, device="cuda")
    assert da.diffattn_fwd_kernel(sh(inp.q), sh(inp.k), sh(inp.v), lam,
                                  inp.subln_w.cuda()) == "diffattn_fwd_bf16_persistent_kernel"
    full = run_gpu(inp, packed=False)
    for s in range(3):
        one = gen()
        a, b = s * T, (s + 1) * T
        one.q, one.k, one.v = one.q[a:b], one.k[a:b], one.v[a:b]
        one.seq_lens, one.cu_seqlens = [T], torch.tensor([0, T], dtype=torch.int32)
        cu = one.cu_seqlens.cuda()
        assert da.diffattn_fwd_kernel(one.q.cuda(), one.k.cuda(), one.v.cuda(), lam, inp.subln_w.cuda(), cu_seqlens=cu,
                                      max_seqlen=T) == "diffattn_fwd_bf16_sm103a_kernel"
        assert torch.equal(run_gpu(one), full[a:b])


# The combined call (lambda kernel, then the forward whose reads of lambda alone
# wait for it) against the two calls, on each forward kernel: the one-item-per-CTA
# bf16 kernel, the persistent one (dense and packed), the fp32 one; lambdas shared
# and per head.
# "tile" and "tile_per_head" fit one wave of CTAs, where the one-item-per-CTA kernel
# forms lambda itself; "tile_waves" (288 CTAs) launches the lambda kernel first.
@pytest.mark.parametrize("case", ["tile", "tile_per_head", "tile_waves", "persistent", "packed", "per_head", "f32"])
def test_fwd_lambda_equals_two_calls_bitwise(case):
    if case == "f32":
        wl, lens = W.WORKLOADS["tiny_f32"], [64]
    elif case == "per_head":
        wl, lens = W.with_overrides(BF, lambda_per_head=True, random_subln=True), [1000, 1000, 1000]
    elif case == "tile_per_head":
        wl, lens = W.with_overrides(BF, num_heads=16, num_kv_heads=4, lambda_per_head=True, random_subln=True), [700]
    else:
        wl = W.with_overrides(BF, num_heads=16, num_kv_heads=4)
        lens = {"tile": [700], "tile_waves": [2300], "persistent": [1000, 1000, 1000],
                "packed": [1000, 40, 2500, 300]}[case]
    inp = W.generate(wl, seed=41, seq_lens=lens)
    t = {n: getattr(inp, n).cuda() for n in ("q", "k", "v", "lambda_q1", "lambda_k1", "lambda_q2", "lambda_k2",
                                             "subln_w", "cu_seqlens")}
    li = da.diffattn_lambda_init(wl.depth)
    vecs = [t["lambda_q1"], t["lambda_k1"], t["lambda_q2"], t["lambda_k2"]]
    packed = case == "packed"
    B, T = len(lens), lens[0]
    sh = (lambda x: x) if packed else (lambda x: x.view(B, T, *x.shape[1:]))  # noqa: E731
    kw = dict(cu_seqlens=t["cu_seqlens"], max_seqlen=max(lens)) if packed else {}
    kern = da.diffattn_fwd_kernel(sh(t["q"]), sh(t["k"]), sh(t["v"]), torch.ones(1, device="cuda"), t["subln_w"],
                                  **kw)
    want_kernel = {"tile": "diffattn_fwd_bf16_sm103a_kernel", "tile_per_head": "diffattn_fwd_bf16_sm103a_kernel",
                   "tile_waves": "diffattn_fwd_bf16_sm103a_kernel", "persistent": "diffattn_fwd_bf16_persistent_kernel",
                   "packed": "diffattn_fwd_bf16_persistent_kernel", "per_head": "diffattn_fwd_bf16_persistent_kernel",
                   "f32": "diffattn_fwd_f32_kernel"}[case]
    assert kern == want_kernel
    lam = da.diffattn_lambda(*vecs, li)
    two = da.diffattn_fwd(sh(t["q"]), sh(t["k"]), sh(t["v"]), lam, li, t["subln_w"], causal=wl.causal, eps=wl.eps,
                          **kw)
    for _ in range(2):  # twice, the second time over the first call's outputs
        one, lam1 = da.diffattn_fwd_lambda(sh(t["q"]), sh(t["k"]), sh(t["v"]), *vecs, li, t["subln_w"],
                                           causal=wl.causal, eps=wl.eps, **kw)
        assert da.diffattn_get_device_status() == 0
        assert torch.equal(lam1, lam)
        assert torch.equal(one, two)


def test_gqa_equals_replicated_bitwise():
    inp = W.generate(BF, seed=32, seq_lens=[400])
    a = run_gpu(inp)
    rep = W.generate(W.with_overrides(BF, num_kv_heads=16), seed=32, seq_lens=[400])
    rep.q, rep.lambda_q1, rep.lambda_k1 = inp.q, inp.lambda_q1, inp.lambda_k1
    rep.lambda_q2, rep.lambda_k2, rep.subln_w = inp.lambda_q2, inp.lambda_k2, inp.subln_w
    rep.k = inp.k.repeat_interleave(4, dim=1)
    rep.v = inp.v.repeat_interleave(4, dim=1)
    assert torch.equal(run_gpu(rep), a)


def test_deterministic():
    inp = W.generate(BF, seed=33, seq_lens=[1000, 24])
    assert torch.equal(run_gpu(inp), run_gpu(inp))


# ------------------------------------------------------------- errors ---

def test_bad_cu_seqlens_reported_and_device_usable():
    inp = W.generate(BF, seed=34, seq_lens=[100, 50])
    t = {n: getattr(inp, n).cuda() for n in ("q", "k", "v", "subln_w")}
    lam = torch.tensor([0.3], device="cuda")
    bad = torch.tensor([0, 120, 150], dtype=torch.int32, device="cuda")  # 120 > max_seqlen 100
    da.diffattn_fwd(t["q"], t["k"], t["v"], lam, 0.2, t["subln_w"], cu_seqlens=bad, max_seqlen=100)
    assert da.diffattn_get_device_status() == 5
    bad2 = torch.tensor([0, 100, 90], dtype=torch.int32, device="cuda")  # not monotone
    da.diffattn_fwd(t["q"], t["k"], t["v"], lam, 0.2, t["subln_w"], cu_seqlens=bad2, max_seqlen=100)
    assert da.diffattn_get_device_status() == 5
    assert da.diffattn_get_device_status() == 0  # cleared by the read
    compare(run_gpu(inp), oracle_out(inp), "bf16")


def test_empty_problem_launches_nothing():
    q = torch.zeros(0, 16, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(0, 4, 128, dtype=torch.bfloat16, device="cuda")
    lam = torch.tensor([0.3], device="cuda")
    w = torch.ones(128, device="cuda")
    out = da.diffattn_fwd(q, k, k, lam, 0.2, w)
    assert out.shape == (0, 16, 128)
    assert da.diffattn_get_device_status() == 0


def test_unsupported_shape_raises():
    q = torch.zeros(10, 2, 64, dtype=torch.bfloat16, device="cuda")  # bf16 with d = 32
    k = torch.zeros(10, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(da.DiffAttnError) as e:
        da.diffattn_fwd(q, k, k, torch.tensor([0.1], device="cuda"), 0.2, torch.ones(64, device="cuda"))
    assert e.value.status == 2
