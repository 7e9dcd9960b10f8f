"""Pins for the fp64 oracle (CPU only).

The pages print no worked example for this path, so the oracle is tied to
things other than itself: closed forms, library special cases (torch's
scaled_dot_product_attention and rms_norm in fp64), a hand-expanded tiny case,
the map-difference brute force, and invariances the definition implies. A
final test plants single mistakes in copies of the oracle source and checks
that every one of them is caught by at least one pin.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as orc
from differential_attention_diffattn_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore")

TOL = 1e-10  # fp64 against fp64: only rounding-order differences remain


# ----------------------------------------------------------------- helpers ---

def _rand_case(seed, H=4, Hkv=2, d=8, lens=(5, 17, 1), causal=True, per_head=False):
    wl = W.Workload("t", "f32", num_heads=H, num_kv_heads=Hkv, d=d, dv=2 * d, depth=3,
                    causal=causal, batch=1, seqlen=1, lambda_per_head=per_head,
                    random_subln=True)
    return W.generate(wl, seed=seed, seq_lens=list(lens))


def _sdpa(qc, kc, v, causal, scale):
    """torch fp64 SDPA per sequence: qc [L, H, d], kc [L, Hkv, d], v [L, Hkv, dv]
    -> [L, H, dv]; grouped heads through enable_gqa (head h reads h // (H/Hkv))."""
    q_ = torch.as_tensor(qc).double().permute(1, 0, 2).unsqueeze(0)
    k_ = torch.as_tensor(kc).double().permute(1, 0, 2).unsqueeze(0)
    v_ = torch.as_tensor(v).double().permute(1, 0, 2).unsqueeze(0)
    o = F.scaled_dot_product_attention(q_, k_, v_, is_causal=causal, scale=scale,
                                       enable_gqa=q_.shape[1] != k_.shape[1])
    return o.squeeze(0).permute(1, 0, 2)


def _rms(x, w, eps):
    x = torch.as_tensor(x).double()
    return F.rms_norm(x, [x.shape[-1]], torch.as_tensor(w).double(), eps)


def _seqs(inp):
    cu = inp.cu_seqlens.tolist()
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


# ---------------------------------------------------------------- the pins ---
# Each pin takes an optional `lib` (another build of the oracle source) so that
# the planted-mistake test can run the same battery against mutants.

def pin_lambda_init(lib=None):
    # l = 1 gives 0.8 - 0.6 = 0.2; the schedule tends to 0.8; the gap to 0.8
    # shrinks by exactly e^-0.3 per layer.
    assert abs(orc.lambda_init(1, lib) - 0.2) < 1e-15
    assert abs(orc.lambda_init(400, lib) - 0.8) < 1e-15
    for l in range(1, 30):
        r = (0.8 - orc.lambda_init(l + 1, lib)) / (0.8 - orc.lambda_init(l, lib))
        assert abs(r - math.exp(-0.3)) < 1e-12


def pin_lambda_special(lib=None):
    z = np.zeros(7)
    # zero vectors: e^0 - e^0 + lambda_init = lambda_init exactly
    assert orc.lambda_values(z, z, z, z, 0.37, lib)[0] == 0.37
    # orthogonal pairs: only q1.k1 = 2 and q2.k2 = 3 survive, cross pairs are 0
    e1, e2 = np.eye(7)[0], np.eye(7)[1]
    got = orc.lambda_values(e1, 2 * e1, e2, 3 * e2, 0.5, lib)[0]
    assert abs(got - (math.exp(2.0) - math.exp(3.0) + 0.5)) < 1e-12
    # several sets are independent
    g = np.random.default_rng(1)
    vs = [g.normal(0, 0.3, (5, 7)) for _ in range(4)]
    many = orc.lambda_values(*vs, 0.1, lib)
    for i in range(5):
        one = orc.lambda_values(*(x[i] for x in vs), 0.1, lib)[0]
        assert abs(many[i] - one) < 1e-15


def pin_hand_example(lib=None):
    """T = 2, d = 1, dv = 2, one head, expanded by hand.
    Scores of component 1 for row 1: [1*0, 1*ln 3] -> softmax [1/4, 3/4];
    component 2 has q2 = 0 -> [1/2, 1/2]. With v0 = [2, 0], v1 = [0, 4]:
    o1 = [0.5, 3], o2 = [1, 2]. lambda = e^(ln 2 * 1) - e^0 + lambda_init(1)
    = 2 - 1 + 0.2 = 1.2, so D1 = [0.5 - 1.2, 3 - 2.4] = [-0.7, 0.6],
    mean D^2 = 0.425. Row 0 sees only key 0: D0 = (1 - 1.2) v0 = [-0.4, 0],
    mean D^2 = 0.08. Output = D / sqrt(mean + eps) * w * (1 - 0.2)."""
    eps = 1e-5
    li = orc.lambda_init(1, lib)
    lam = orc.lambda_values([math.log(2.0)], [1.0], [0.0], [0.0], li, lib)
    assert abs(lam[0] - 1.2) < 1e-14
    q = np.array([[[0.0, 0.0]], [[1.0, 0.0]]])
    k = np.array([[[0.0, 5.0]], [[math.log(3.0), 7.0]]])
    v = np.array([[[2.0, 0.0]], [[0.0, 4.0]]])
    w = np.array([1.0, 0.5])
    got = orc.forward_rows([0, 2], q, k, v, lam, li, w, eps, True, lib=lib)
    want1 = np.array([-0.7, 0.6]) / math.sqrt(0.425 + eps) * w * 0.8
    want0 = np.array([-0.4, 0.0]) / math.sqrt(0.08 + eps) * w * 0.8
    np.testing.assert_allclose(got[1, 0], want1, atol=1e-13, rtol=0)
    np.testing.assert_allclose(got[0, 0], want0, atol=1e-13, rtol=0)


def pin_lambda_zero_is_sdpa(lib=None):
    """lambda = 0: the output is RMSNorm(causal softmax attention of (Q1, K1, V))
    * w * (1 - lambda_init), checked against torch's SDPA and rms_norm."""
    for causal, (H, Hkv) in [(True, (4, 2)), (False, (4, 2)), (True, (3, 3)), (True, (4, 1))]:
        inp = _rand_case(11, H=H, Hkv=Hkv, d=8, lens=(9, 1, 23), causal=causal)
        d, li = inp.wl.d, 0.3
        got = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, 0.0, li, inp.subln_w,
                               inp.wl.eps, causal, lib=lib)
        for a, b in _seqs(inp):
            att = _sdpa(inp.q[a:b, :, :d], inp.k[a:b, :, :d], inp.v[a:b], causal, d ** -0.5)
            want = _rms(att, inp.subln_w, inp.wl.eps) * (1 - li)
            np.testing.assert_allclose(got[a:b], want.numpy(), atol=TOL, rtol=0)


def pin_equal_components(lib=None):
    """Q1 = Q2 and K1 = K2: both maps coincide, so the pre-norm output is
    (1 - lambda) * attention(Q1, K1, V), for any lambda (also lambda > 1)."""
    inp = _rand_case(12, H=4, Hkv=2, d=8, lens=(13, 30))
    d = inp.wl.d
    q, k = inp.q.clone(), inp.k.clone()
    q[:, :, d:] = q[:, :, :d]
    k[:, :, d:] = k[:, :, :d]
    for lam in (0.35, 1.7, -0.4):
        li = 0.61
        got = orc.forward_rows(inp.cu_seqlens, q, k, inp.v, lam, li, inp.subln_w, inp.wl.eps,
                               True, lib=lib)
        for a, b in _seqs(inp):
            att = _sdpa(q[a:b, :, :d], k[a:b, :, :d], inp.v[a:b], True, d ** -0.5)
            want = _rms((1 - lam) * att, inp.subln_w, inp.wl.eps) * (1 - li)
            np.testing.assert_allclose(got[a:b], want.numpy(), atol=TOL, rtol=0)


def pin_row0_closed_form(lib=None):
    """Causal row 0 of every sequence sees only key 0: D = (1 - lambda) V[0]."""
    inp = _rand_case(13, H=4, Hkv=2, d=8, lens=(7, 3, 1))
    li = 0.45
    lam = np.array([0.2, 0.9, 1.3, -0.1])
    got = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, lam, li, inp.subln_w,
                           inp.wl.eps, True, lib=lib)
    for a, _ in _seqs(inp):
        for h in range(4):
            v0 = inp.v[a, h // 2].double().numpy()
            dd = (1 - lam[h]) * v0
            want = dd / np.sqrt(np.mean(dd ** 2) + inp.wl.eps) * inp.subln_w.double().numpy() * (1 - li)
            np.testing.assert_allclose(got[a, h], want, atol=TOL, rtol=0)


def pin_uniform_scores(lib=None):
    """Q = 0: every score is 0, each softmax is uniform over the visible keys,
    so row i gets D = (1 - lambda) * mean_{j <= i} V[j]."""
    inp = _rand_case(14, H=2, Hkv=1, d=8, lens=(19,))
    q = torch.zeros_like(inp.q)
    lam, li = 0.6, 0.3
    got = orc.forward_rows(inp.cu_seqlens, q, inp.k, inp.v, lam, li, inp.subln_w, inp.wl.eps,
                           True, lib=lib)
    vv = inp.v[:, 0].double().numpy()
    cmean = np.cumsum(vv, axis=0) / np.arange(1, vv.shape[0] + 1)[:, None]
    dd = (1 - lam) * cmean
    want = dd / np.sqrt(np.mean(dd ** 2, axis=-1, keepdims=True) + inp.wl.eps) * inp.subln_w.double().numpy() * (1 - li)
    for h in range(2):
        np.testing.assert_allclose(got[:, h], want, atol=TOL, rtol=0)


def pin_map_form(lib=None):
    """The C oracle (output-difference form) equals the NumPy map-difference
    brute force on random shapes, causal and not, grouped heads, packed."""
    cases = [dict(H=4, Hkv=2, d=8, lens=(5, 17, 1)), dict(H=2, Hkv=2, d=16, lens=(33,)),
             dict(H=6, Hkv=3, d=4, lens=(2, 9), causal=False),
             dict(H=4, Hkv=1, d=8, lens=(12, 12), per_head=True)]
    for i, c in enumerate(cases):
        inp = _rand_case(20 + i, **c)
        li = orc.lambda_init(5, lib)
        lam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, li, lib)
        causal = c.get("causal", True)
        a = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, lam, li, inp.subln_w,
                             inp.wl.eps, causal, lib=lib)
        b = orc.forward_map_form(inp.cu_seqlens, inp.q, inp.k, inp.v, lam, li, inp.subln_w,
                                 inp.wl.eps, causal)
        np.testing.assert_allclose(a, b, atol=1e-12, rtol=0)


def pin_scale_invariance(lib=None):
    """With eps = 0 the norm removes any positive scale of V: y(cV) = y(V)."""
    inp = _rand_case(15, H=2, Hkv=2, d=8, lens=(11,))
    a = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, 0.7, 0.2, inp.subln_w, 0.0, True, lib=lib)
    b = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v.double() * 3.5, 0.7, 0.2, inp.subln_w, 0.0, True, lib=lib)
    np.testing.assert_allclose(a, b, atol=TOL, rtol=0)


def pin_gqa_equals_replicated(lib=None):
    """Grouped heads equal explicitly replicated key/value heads."""
    inp = _rand_case(16, H=6, Hkv=2, d=8, lens=(10, 4))
    a = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, 0.4, 0.3, inp.subln_w, 1e-5, True, lib=lib)
    k_rep = inp.k.repeat_interleave(3, dim=1)
    v_rep = inp.v.repeat_interleave(3, dim=1)
    b = orc.forward_rows(inp.cu_seqlens, inp.q, k_rep, v_rep, 0.4, 0.3, inp.subln_w, 1e-5, True, lib=lib)
    np.testing.assert_allclose(a, b, atol=TOL, rtol=0)


def pin_packed_equals_separate(lib=None):
    """A packed batch equals each sequence run on its own."""
    inp = _rand_case(17, H=2, Hkv=1, d=8, lens=(6, 1, 14))
    full = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, 0.4, 0.3, inp.subln_w, 1e-5, True, lib=lib)
    for a, b in _seqs(inp):
        one = orc.forward_rows([0, b - a], inp.q[a:b], inp.k[a:b], inp.v[a:b], 0.4, 0.3,
                               inp.subln_w, 1e-5, True, lib=lib)
        np.testing.assert_allclose(full[a:b], one, atol=TOL, rtol=0)


def pin_head_permutation(lib=None):
    """Permuting diff heads (with their lambda) permutes the output heads."""
    inp = _rand_case(18, H=4, Hkv=4, d=8, lens=(9,))
    lam = np.array([0.1, 0.5, 0.9, 1.4])
    perm = [2, 0, 3, 1]
    a = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, lam, 0.3, inp.subln_w, 1e-5, True, lib=lib)
    b = orc.forward_rows(inp.cu_seqlens, inp.q[:, perm], inp.k[:, perm], inp.v[:, perm], lam[perm],
                         0.3, inp.subln_w, 1e-5, True, lib=lib)
    np.testing.assert_allclose(a[:, perm], b, atol=TOL, rtol=0)


def pin_rows_subset(lib=None):
    """Computing selected rows gives the same numbers as the full output."""
    inp = _rand_case(19, H=4, Hkv=2, d=8, lens=(7, 20))
    full = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, 0.4, 0.3, inp.subln_w, 1e-5, True, lib=lib)
    tok = np.array([0, 6, 7, 26, 13])
    hd = np.array([3, 0, 1, 2, 2])
    part = orc.forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, 0.4, 0.3, inp.subln_w, 1e-5, True,
                            rows=(tok, hd), lib=lib)
    np.testing.assert_array_equal(part, full[tok, hd])


def pin_bottom_right_mask(lib=None):
    """New queries at the end of a cached sequence: the oracle rows of the last
    q_len positions equal the map form with the bottom-right mask
    triu(-inf, 1 + src_len - tgt_len) of the FlashDiffAttention review snippet
    (tgt_len = q_len queries against src_len = L keys), written out in NumPy."""
    g = np.random.default_rng(7)
    L, ql, H, Hkv, d = 11, 4, 4, 2, 8
    q_new = g.normal(size=(ql, H, 2 * d))
    k = g.normal(size=(L, Hkv, 2 * d))
    v = g.normal(size=(L, Hkv, 2 * d))
    w = g.uniform(0.5, 1.5, size=2 * d)
    lam, li, eps = np.array([0.3, 0.9, -0.2, 1.4]), 0.55, 1e-5
    q_full = np.zeros((L, H, 2 * d))
    q_full[L - ql:] = q_new
    tt = np.repeat(np.arange(L - ql, L, dtype=np.int32), H)
    hh = np.tile(np.arange(H, dtype=np.int32), ql)
    got = orc.forward_rows([0, L], q_full, k, v, lam, li, w, eps, True, rows=(tt, hh), lib=lib).reshape(ql, H, -1)
    mask = np.triu(np.full((ql, L), -np.inf), 1 + L - ql)
    for h in range(H):
        kv = h // (H // Hkv)
        maps = []
        for c in range(2):
            a = q_new[:, h, c * d:(c + 1) * d] @ k[:, kv, c * d:(c + 1) * d].T * d ** -0.5 + mask
            a = np.exp(a - a.max(axis=1, keepdims=True))
            maps.append(a / a.sum(axis=1, keepdims=True))
        o = (maps[0] - lam[h] * maps[1]) @ v[:, kv, :]
        want = o / np.sqrt(np.mean(o ** 2, axis=-1, keepdims=True) + eps) * w * (1 - li)
        np.testing.assert_allclose(got[:, h], want, atol=TOL, rtol=0)


PINS = [pin_lambda_init, pin_lambda_special, pin_hand_example, pin_lambda_zero_is_sdpa,
        pin_equal_components, pin_row0_closed_form, pin_uniform_scores, pin_map_form,
        pin_scale_invariance, pin_gqa_equals_replicated, pin_packed_equals_separate,
        pin_head_permutation, pin_rows_subset, pin_bottom_right_mask]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# Single planted mistakes in a copy of the oracle source: (original, mutant).
MUTATIONS = [
    ("y[e] = o1[e] - lam * o2[e];", "y[e] = o1[e] + lam * o2[e];"),          # sign of lambda term
    ("y[e] = o1[e] - lam * o2[e];", "y[e] = o1[e] - o2[e];"),                # lambda dropped
    ("y[e] = o1[e] - lam * o2[e];", "y[e] = o1[e] - lam * o1[e];"),          # second map dropped
    ("1.0 / sqrt((double)d)", "1.0 / sqrt((double)dv)"),                    # scale on dv
    ("const int g = h / group;", "const int g = h % Hkv;"),                  # GQA mapping
    ("causal ? i + 1 : len", "len"),                                          # mask dropped
    ("* (1.0 - lambda_init)", ""),                                            # post-norm factor
    ("ms /= (double)dv;", "ms /= (double)d;"),                                # RMS extent
    ("sqrt(ms + eps)", "sqrt(ms)"),                                           # eps dropped
    ("* (size_t)(2 * d) + (size_t)c * d;", "* (size_t)(2 * d);"),             # K2 read as K1
    ("const double* qr = qrow + (size_t)c * d;", "const double* qr = qrow;"),  # Q2 read as Q1
    ("v + ((size_t)(start + j) * Hkv + g)", "v + ((size_t)(start + n_keys - 1 - j) * Hkv + g)"),  # V order
    ("out[i] = exp(a) - exp(b) + lambda_init;", "out[i] = exp(a) - exp(b) - lambda_init;"),
    ("lk1[(size_t)i * d + e];", "lk2[(size_t)i * d + e];"),                    # cross pairing
    ("exp(-0.3 * (double)(depth - 1))", "exp(-0.3 * (double)depth)"),         # depth index
]


def test_planted_mistakes_are_caught(tmp_path):
    src = open(orc._SRC).read()
    survivors = []
    for i, (a, b) in enumerate(MUTATIONS):
        assert src.count(a) == 1, a
        mutant = tmp_path / f"m{i}.c"
        mutant.write_text(src.replace(a, b))
        so = orc.build(force=True, src=str(mutant), out=str(tmp_path / f"libm{i}.so"))
        lib = orc._load(so)
        caught = False
        for pin in PINS:
            try:
                pin(lib)
            except (AssertionError, ValueError, FloatingPointError):
                caught = True
                break
        if not caught:
            survivors.append(b)
    assert not survivors, f"mutants not caught by any pin: {survivors}"


# ------------------------------------------------------------ regression ---

def test_golden_tiny_f32():
    """The committed oracle outputs for the tiny fp32 workload (written by
    tests/golden/make_golden.py, which calls only the oracle) still hold."""
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny_f32_seed0.txt")
    data = np.loadtxt(path)
    inp = W.generate(W.WORKLOADS["tiny_f32"], seed=0)
    out = orc.forward(inp)
    tok, hd = data[:, 0].astype(int), data[:, 1].astype(int)
    np.testing.assert_allclose(out[tok, hd], data[:, 2:], atol=1e-12, rtol=0)
