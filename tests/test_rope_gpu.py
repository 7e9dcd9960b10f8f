"""GPU parity of the rotary embedding: the cos / sin tables, the rotation of q
and k in both placements the pages use (whole 2d-wide row, half-split pairs;
every d-wide component, interleaved pairs) and the third combination, with
positions from the dense layout, cu_seqlens or an explicit array, in place and
out of place, and the rotation followed by the attention, against the fp64
oracles (oracle/rope.py, then the attention oracle)."""
import numpy as np
import pytest
import torch

import differential_attention_diffattn_gb300 as da
from differential_attention_diffattn_gb300 import workloads as W
from oracle import rope as orope
from oracle import oracle as orc

from gpu_util import compare

pytestmark = pytest.mark.gpu

PLACEMENTS = [(128, False), (64, True), (64, False), (128, True)]  # (rot_dim, interleaved) with d = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    da.build()
    da.load_library()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("theta,n_pos,rot", [(10000.0, 16384, 64), (500000.0, 4096, 128), (10000.0, 7, 8)])
def test_tables_match_oracle(theta, n_pos, rot):
    cos, sin = da.diffattn_rope_tables(theta, n_pos, rot)
    wc, ws = orope.tables(theta, n_pos, rot)
    # fp64 on the device, one rounding to fp32: within half an fp32 ulp of values <= 1
    assert np.abs(cos.cpu().numpy() - wc).max() <= 6e-8
    assert np.abs(sin.cpu().numpy() - ws).max() <= 6e-8


def _check_rotation(got, x, pos, rot, inter, theta, n_pos):
    wc, ws = orope.tables(theta, n_pos, rot)
    want = orope.apply(x.double().cpu().numpy(), pos, wc, ws, rot, inter)
    g = got.double().cpu().numpy()
    if got.dtype == torch.bfloat16:
        # fp32 arithmetic then one round-to-nearest to bf16 (half an ulp = 2^-9 relative)
        bound = 2.0 ** -8 * np.abs(want) + 1e-5
    else:
        bound = 1e-6 * (np.abs(x.double().cpu().numpy()).max() + 1.0)
    err = np.abs(g - want)
    assert (err <= bound).all(), (float(err.max()), np.unravel_index(np.argmax(err - bound), err.shape))


@pytest.mark.parametrize("rot,inter", PLACEMENTS)
@pytest.mark.parametrize("source", ["dense", "cu_seqlens", "positions"])
def test_rotation_matches_oracle(rot, inter, source):
    g = torch.Generator().manual_seed(11)
    B, T, H, Hkv, d = 2, 300, 8, 2, 64
    q = torch.randn(B * T, H, 2 * d, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B * T, Hkv, 2 * d, generator=g).to(torch.bfloat16).cuda()
    n_pos = 4096
    cos, sin = da.diffattn_rope_tables(10000.0, n_pos, rot)
    if source == "dense":
        qo, ko = da.diffattn_rope_qk(q.view(B, T, H, 2 * d), k.view(B, T, Hkv, 2 * d), cos, sin, rot, inter)
        qo, ko = qo.view(B * T, H, 2 * d), ko.view(B * T, Hkv, 2 * d)
        pos = np.tile(np.arange(T), B)
    elif source == "cu_seqlens":
        lens = [1, 250, 0, 349]
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32).cuda()
        qo, ko = da.diffattn_rope_qk(q, k, cos, sin, rot, inter, cu_seqlens=cu)
        pos = orope.positions_from_cu_seqlens(cu.cpu().numpy())
    else:
        pos = np.random.default_rng(3).integers(0, n_pos, B * T)
        qo, ko = da.diffattn_rope_qk(q, k, cos, sin, rot, inter,
                                     positions=torch.tensor(pos, dtype=torch.int32).cuda())
    assert da.diffattn_get_device_status() == 0
    _check_rotation(qo, q, pos, rot, inter, 10000.0, n_pos)
    _check_rotation(ko, k, pos, rot, inter, 10000.0, n_pos)


def test_in_place_fp32_and_q_only():
    g = torch.Generator().manual_seed(12)
    T, H, d = 77, 3, 16
    x = torch.randn(T, H, 2 * d, generator=g).cuda()
    x0 = x.clone()
    cos, sin = da.diffattn_rope_tables(10000.0, 128, 2 * d)
    da.diffattn_rope_qk(x, None, cos, sin, 2 * d, False, q_out=x)
    assert da.diffattn_get_device_status() == 0
    _check_rotation(x, x0, np.arange(T), 2 * d, False, 10000.0, 128)


def test_position_outside_tables_is_reported():
    T, H, Hkv, d = 40, 2, 1, 64
    g = torch.Generator().manual_seed(13)
    q = torch.randn(T, H, 2 * d, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(T, Hkv, 2 * d, generator=g).to(torch.bfloat16).cuda()
    cos, sin = da.diffattn_rope_tables(10000.0, 32, d)
    pos = np.arange(T) % 32
    pos[7] = 32                      # one past the tables
    pos[9] = -1
    qo, ko = da.diffattn_rope_qk(q, k, cos, sin, d, True, positions=torch.tensor(pos, dtype=torch.int32).cuda())
    assert da.diffattn_get_device_status() == da._lib.ERR_BAD_POSITIONS
    assert da.diffattn_get_device_status() == 0          # read and cleared
    assert torch.equal(qo[7], q[7]) and torch.equal(ko[9], k[9])   # passed through unrotated
    ok = np.setdiff1d(np.arange(T), [7, 9])
    _check_rotation(qo[ok], q[ok], pos[ok], d, True, 10000.0, 32)


@pytest.mark.parametrize("rot,inter", [(128, False), (64, True)])
def test_rope_then_attention_matches_oracle(rot, inter):
    """The two placements end to end: rotate q and k on the GPU, run the forward;
    the oracle rotates in fp64 and runs its own forward."""
    wl = W.with_overrides(W.WORKLOADS["b2_t512_gqa"], random_subln=True)
    inp = W.generate(wl, seed=21, seq_lens=[700, 129, 195])
    theta, n_pos = 10000.0, 1024
    cos, sin = da.diffattn_rope_tables(theta, n_pos, rot)
    cu = inp.cu_seqlens.cuda()
    qr, kr = da.diffattn_rope_qk(inp.q.cuda(), inp.k.cuda(), cos, sin, rot, inter, cu_seqlens=cu)
    li = da.diffattn_lambda_init(wl.depth)
    lam = da.diffattn_lambda(*(x.cuda() for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)), li)
    y = da.diffattn_fwd(qr, kr, inp.v.cuda(), lam, li, inp.subln_w.cuda(), causal=True, cu_seqlens=cu,
                        max_seqlen=inp.max_seqlen, eps=wl.eps)
    assert da.diffattn_get_device_status() == 0
    wc, ws = orope.tables(theta, n_pos, rot)
    pos = orope.positions_from_cu_seqlens(inp.cu_seqlens.numpy())
    q64 = orope.apply(inp.q.double().numpy(), pos, wc, ws, rot, inter)
    k64 = orope.apply(inp.k.double().numpy(), pos, wc, ws, rot, inter)
    oli = orc.lambda_init(wl.depth)
    olam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, oli)
    want = orc.forward_rows(inp.cu_seqlens, q64, k64, inp.v, olam, oli, inp.subln_w, wl.eps, True)
    compare(y, want, "bf16")


def _fused_case(wl, seq_lens, seed, dense):
    inp = W.generate(wl, seed=seed, seq_lens=seq_lens)
    B, T = len(inp.seq_lens), inp.seq_lens[0]
    sh = (lambda x: x.cuda().view(B, T, *x.shape[1:])) if dense else (lambda x: x.cuda())
    kw = {} if dense else dict(cu_seqlens=inp.cu_seqlens.cuda(), max_seqlen=inp.max_seqlen)
    li = da.diffattn_lambda_init(wl.depth)
    lam = da.diffattn_lambda(*(x.cuda() for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)), li)
    return inp, sh, kw, li, lam


# A dense 4 x 1024 batch (its plain forward takes the persistent kernel, the
# fused one the one-item-per-CTA kernel: the two give the same bits) and three
# packed sequences (both on the one-item-per-CTA kernel).
KERNEL_CASES = [("dense_4x1024", [1024] * 4, True), ("packed_3", [700, 129, 195], False)]


@pytest.mark.parametrize("rot,inter", PLACEMENTS)
@pytest.mark.parametrize("case,lens,dense", KERNEL_CASES)
def test_fused_rotation_equals_separate_pass(rot, inter, case, lens, dense):
    """q rotated inside the forward kernel against q rotated by the separate
    pass and then the plain forward: the same bits (the same expressions with the
    same explicit roundings, the same tables)."""
    wl = W.with_overrides(W.WORKLOADS["b2_t512_gqa"], random_subln=True)
    inp, sh, kw, li, lam = _fused_case(wl, lens, 31, dense)
    q, k, v, w = sh(inp.q), sh(inp.k), sh(inp.v), inp.subln_w.cuda()
    cos, sin = da.diffattn_rope_tables(10000.0, 2048, rot)
    cu = kw.get("cu_seqlens")
    qr, kr = da.diffattn_rope_qk(q, k, cos, sin, rot, inter, cu_seqlens=cu)
    kr_only = da.diffattn_rope_k(k, cos, sin, rot, inter, cu_seqlens=cu)
    assert torch.equal(kr_only, kr)
    ref = da.diffattn_fwd(qr, kr, v, lam, li, w, causal=True, eps=wl.eps, **kw)
    got = da.diffattn_fwd_rope_q(q, kr_only, v, lam, li, w, cos, sin, rot, inter, causal=True, eps=wl.eps, **kw)
    assert da.diffattn_get_device_status() == 0
    assert torch.equal(got, ref)


@pytest.mark.parametrize("rot,inter", [(128, False), (64, True)])
def test_fused_rope_then_attention_matches_oracle(rot, inter):
    """The two placements end to end through the fused entry: k rotated by the
    separate pass, q inside the forward; the oracle rotates in fp64 and runs its
    own forward."""
    wl = W.with_overrides(W.WORKLOADS["b2_t512_gqa"], random_subln=True)
    inp = W.generate(wl, seed=21, seq_lens=[700, 129, 195])
    theta, n_pos = 10000.0, 1024
    cos, sin = da.diffattn_rope_tables(theta, n_pos, rot)
    cu = inp.cu_seqlens.cuda()
    kr = da.diffattn_rope_k(inp.k.cuda(), cos, sin, rot, inter, cu_seqlens=cu)
    li = da.diffattn_lambda_init(wl.depth)
    lam = da.diffattn_lambda(*(x.cuda() for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)), li)
    y = da.diffattn_fwd_rope_q(inp.q.cuda(), kr, inp.v.cuda(), lam, li, inp.subln_w.cuda(), cos, sin, rot, inter,
                               causal=True, cu_seqlens=cu, max_seqlen=inp.max_seqlen, eps=wl.eps)
    assert da.diffattn_get_device_status() == 0
    wc, ws = orope.tables(theta, n_pos, rot)
    pos = orope.positions_from_cu_seqlens(inp.cu_seqlens.numpy())
    q64 = orope.apply(inp.q.double().numpy(), pos, wc, ws, rot, inter)
    k64 = orope.apply(inp.k.double().numpy(), pos, wc, ws, rot, inter)
    oli = orc.lambda_init(wl.depth)
    olam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, oli)
    want = orc.forward_rows(inp.cu_seqlens, q64, k64, inp.v, olam, oli, inp.subln_w, wl.eps, True)
    compare(y, want, "bf16")


@pytest.mark.parametrize("case,lens,dense", KERNEL_CASES)
def test_fused_rotation_reports_positions_past_the_tables(case, lens, dense):
    wl = W.WORKLOADS["b2_t512_gqa"]
    inp, sh, kw, li, lam = _fused_case(wl, lens, 32, dense)
    q, k, v, w = sh(inp.q), sh(inp.k), sh(inp.v), inp.subln_w.cuda()
    cos, sin = da.diffattn_rope_tables(10000.0, 600, 64)  # shorter than the longest sequence
    da.diffattn_fwd_rope_q(q, k, v, lam, li, w, cos, sin, 64, True, causal=True, eps=wl.eps, **kw)
    assert da.diffattn_get_device_status() == da._lib.ERR_BAD_POSITIONS
    assert da.diffattn_get_device_status() == 0


def test_fused_rotation_non_causal_per_head_lambda_and_k_positions():
    """The fused entry with a non-causal mask, a lambda per head and a random
    weight, k rotated by explicit positions (those of the packed layout), against
    the oracle."""
    wl = W.with_overrides(W.WORKLOADS["b2_t512_gqa"], causal=False, lambda_per_head=True, random_subln=True)
    inp = W.generate(wl, seed=33, seq_lens=[300, 77, 129])
    rot, inter, theta, n_pos = 64, False, 10000.0, 512
    cos, sin = da.diffattn_rope_tables(theta, n_pos, rot)
    pos = orope.positions_from_cu_seqlens(inp.cu_seqlens.numpy())
    kr = da.diffattn_rope_k(inp.k.cuda(), cos, sin, rot, inter,
                            positions=torch.tensor(pos, dtype=torch.int32).cuda())
    li = da.diffattn_lambda_init(wl.depth)
    lam = da.diffattn_lambda(*(x.cuda() for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)), li)
    assert lam.numel() == wl.num_heads
    y = da.diffattn_fwd_rope_q(inp.q.cuda(), kr, inp.v.cuda(), lam, li, inp.subln_w.cuda(), cos, sin, rot, inter,
                               causal=False, cu_seqlens=inp.cu_seqlens.cuda(), max_seqlen=inp.max_seqlen, eps=wl.eps)
    assert da.diffattn_get_device_status() == 0
    wc, ws = orope.tables(theta, n_pos, rot)
    q64 = orope.apply(inp.q.double().numpy(), pos, wc, ws, rot, inter)
    k64 = orope.apply(inp.k.double().numpy(), pos, wc, ws, rot, inter)
    oli = orc.lambda_init(wl.depth)
    olam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, oli)
    want = orc.forward_rows(inp.cu_seqlens, q64, k64, inp.v, olam, oli, inp.subln_w, wl.eps, False)
    compare(y, want, "bf16")
