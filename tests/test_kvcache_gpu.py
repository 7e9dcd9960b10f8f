"""GPU parity of the cache forward (decode / short query blocks) against the
fp64 oracle, element by element, including the split-merge edge cases."""
import numpy as np
import pytest
import torch

import differential_attention_diffattn_gb300 as da
from differential_attention_diffattn_gb300 import workloads as W

from gpu_util import compare, oracle_kv, run_gpu_kv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    da.build()
    da.load_library()
    torch.cuda.set_device(0)


def kvw(**kw):
    base = dict(num_heads=16, num_kv_heads=4, d=64, dv=128, depth=12, batch=3, q_len=1, capacity=1000)
    base.update(kw)
    return W.KvWorkload("t", **base)


# R = q_len * H / Hkv query rows per kv head: 1 ... 32, powers of two or not
@pytest.mark.parametrize("H,Hkv,ql", [(16, 4, 1), (4, 4, 1), (8, 4, 1), (16, 16, 2), (16, 4, 2), (16, 4, 4),
                                      (16, 1, 1), (8, 8, 2), (16, 4, 3), (12, 4, 5), (4, 4, 7), (16, 4, 8),
                                      (32, 1, 1)])
def test_rows_per_kv_head(H, Hkv, ql):
    wl = kvw(num_heads=H, num_kv_heads=Hkv, q_len=ql)
    inp = W.generate_kv(wl, seed=H + Hkv + ql, lengths=[1000, 517, ql])
    compare(run_gpu_kv(inp), oracle_kv(inp), "bf16")


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 16])
def test_forced_splits(splits):
    inp = W.generate_kv(kvw(batch=2, capacity=2000), seed=40 + splits, lengths=[2000, 65])
    compare(run_gpu_kv(inp, num_splits=splits), oracle_kv(inp), "bf16")


def test_non_causal_and_per_head_lambda():
    wl = kvw(q_len=4, causal=False, lambda_per_head=True, random_subln=True)
    inp = W.generate_kv(wl, seed=50, lengths=[1000, 300, 4])
    compare(run_gpu_kv(inp), oracle_kv(inp), "bf16")


def test_full_caches_without_lengths():
    inp = W.generate_kv(kvw(batch=2, capacity=777), seed=51)
    compare(run_gpu_kv(inp, use_seqlens=False), oracle_kv(inp), "bf16")


@pytest.mark.parametrize("name", ["decode_b8_c16384", "decode_b16_q4_ragged"])
def test_cache_workloads(name):
    inp = W.generate_kv(W.KV_WORKLOADS[name], seed=0)
    got = run_gpu_kv(inp)
    assert torch.isfinite(got.float()).all()
    b_sel = [0, inp.wl.batch // 2, inp.wl.batch - 1]
    compare(got[b_sel], oracle_kv(inp, b_sel), "bf16")


def test_bad_cache_lengths_reported():
    inp = W.generate_kv(kvw(batch=2, q_len=2), seed=52, lengths=[1000, 1])  # 1 < q_len
    with pytest.raises(AssertionError):
        run_gpu_kv(inp)
    assert da.diffattn_get_device_status() == 0
    good = W.generate_kv(kvw(batch=2, q_len=2), seed=52, lengths=[1000, 2])
    compare(run_gpu_kv(good), oracle_kv(good), "bf16")


def test_unsupported_rows():
    inp = W.generate_kv(kvw(q_len=9), seed=53)  # 9 * 4 = 36 rows per kv head (at most 32)
    with pytest.raises(da.DiffAttnError) as e:
        run_gpu_kv(inp)
    assert e.value.status == 2


def test_deterministic_and_workspace_reuse():
    inp = W.generate_kv(kvw(batch=2), seed=54, lengths=[999, 400])
    a = run_gpu_kv(inp)
    b = run_gpu_kv(inp)
    assert torch.equal(a, b)


def test_poisoned_rows_beyond_lengths_are_never_used():
    # cache rows past each length (read by the last tile of a split) hold NaN and
    # Inf: a zero probability times NaN would still be NaN
    inp = W.generate_kv(kvw(batch=3, q_len=2), seed=55, lengths=[1000, 517, 70])
    for b, L in enumerate(inp.cache_seqlens.tolist()):
        inp.k_cache[b, L:] = float("nan")
        inp.v_cache[b, L::2] = float("nan")
        inp.v_cache[b, L + 1::2] = float("inf")
    got = run_gpu_kv(inp)
    assert torch.isfinite(got.float()).all()
    compare(got, oracle_kv(inp), "bf16")


def test_split_past_the_visible_keys_of_early_rows():
    # 4 new tokens, chunks of 256 keys: with L = 258 the split [256, 258) sees no
    # key visible to the first new query (position 254): an empty partial
    inp = W.generate_kv(kvw(batch=3, q_len=4), seed=56, lengths=[258, 130, 1000])
    compare(run_gpu_kv(inp, num_splits=4), oracle_kv(inp), "bf16")


def test_ragged_lengths_library_splits():
    # library-planned splits over ragged caches: lengths from one tile to the
    # whole cache, so most splits of the short sequences hold no key
    inp = W.generate_kv(kvw(batch=6, capacity=4000, q_len=2), seed=57, lengths=[4000, 10, 2500, 700, 64, 3999])
    compare(run_gpu_kv(inp), oracle_kv(inp), "bf16")


def test_more_groups_than_resident_ctas():
    # 200 sequences x 4 kv heads: more (sequence, kv head) groups than resident
    # split CTAs, so the plan takes one split each over more than one wave
    rng = np.random.default_rng(58)
    lengths = rng.integers(1, 301, 200).tolist()
    inp = W.generate_kv(kvw(batch=200, capacity=300), seed=58, lengths=lengths)
    compare(run_gpu_kv(inp), oracle_kv(inp), "bf16")


@pytest.mark.parametrize("name", ["decode_b8_c16384", "decode_b16_q4_ragged"])
def test_cache_workloads_with_host_lengths(name):
    """The split plan from a host copy of the lengths (7 splits on the ragged
    batch, 8 on the uniform one, against 4 and 9 from the shape alone): the same
    results within the tolerance, on sampled sequences against the oracle."""
    inp = W.generate_kv(W.KV_WORKLOADS[name], seed=0)
    got = run_gpu_kv(inp, host_seqlens=True)
    ref = run_gpu_kv(inp)
    compare(got, ref.double().cpu().numpy(), "bf16")
    b_sel = [0, inp.wl.batch // 2, inp.wl.batch - 1]
    compare(got[b_sel], oracle_kv(inp, b_sel), "bf16")


def test_host_lengths_on_mixed_batch():
    # one long sequence among short ones: the plan spreads the long one over many splits
    inp = W.generate_kv(kvw(batch=4, capacity=4096), seed=52, lengths=[100, 200, 4096, 30])
    compare(run_gpu_kv(inp, host_seqlens=True), oracle_kv(inp), "bf16")


@pytest.mark.parametrize("hint", ["capacity", "q_len", "reversed"])
def test_host_lengths_are_only_a_plan_hint(hint):
    """Host lengths that disagree with the device's change only the split count:
    the kernels use the device lengths, so the results stay those of the oracle."""
    inp = W.generate_kv(kvw(batch=4, capacity=3000, q_len=2), seed=53, lengths=[3000, 40, 1700, 2])
    wl = inp.wl
    wrong = {"capacity": [wl.capacity] * 4, "q_len": [wl.q_len] * 4,
             "reversed": inp.cache_seqlens.flip(0).tolist()}[hint]
    li = da.diffattn_lambda_init(wl.depth)
    lam = da.diffattn_lambda(inp.lambda_q1.cuda(), inp.lambda_k1.cuda(), inp.lambda_q2.cuda(), inp.lambda_k2.cuda(),
                             li)
    y = da.diffattn_fwd_kvcache(inp.q.cuda(), inp.k_cache.cuda(), inp.v_cache.cuda(), lam, li, inp.subln_w.cuda(),
                                cache_seqlens=inp.cache_seqlens.cuda(), causal=wl.causal, eps=wl.eps,
                                host_seqlens=wrong)
    assert da.diffattn_get_device_status() == 0
    compare(y, oracle_kv(inp), "bf16")


# diffattn_fwd_kvcache_lambda against diffattn_lambda + diffattn_fwd_kvcache: the
# same bits for lambda and for the output (shared and per-head lambda, a forced
# split count and the library's plan, both cache workloads' shapes).
@pytest.mark.parametrize("case", ["shared", "per_head", "splits3", "decode_b8_c16384", "decode_b16_q4_ragged"])
def test_kvcache_lambda_equals_two_calls_bitwise(case):
    if case in W.KV_WORKLOADS:
        inp = W.generate_kv(W.KV_WORKLOADS[case], seed=61)
        splits = 0
    else:
        wl = kvw(q_len=2, lambda_per_head=case == "per_head", random_subln=True)
        inp = W.generate_kv(wl, seed=60, lengths=[1000, 517, 2])
        splits = 3 if case == "splits3" else 0
    wl = inp.wl
    dev = "cuda"
    li = da.diffattn_lambda_init(wl.depth)
    vecs = [x.to(dev) for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)]
    args = (inp.q.to(dev), inp.k_cache.to(dev), inp.v_cache.to(dev))
    lens = inp.cache_seqlens.to(dev)
    w = inp.subln_w.to(dev)
    lam = da.diffattn_lambda(*vecs, li)
    two = da.diffattn_fwd_kvcache(*args, lam, li, w, cache_seqlens=lens, causal=wl.causal, eps=wl.eps,
                                  num_splits=splits)
    for _ in range(2):  # twice, the second time over the first call's outputs
        one, lam1 = da.diffattn_fwd_kvcache_lambda(*args, *vecs, li, w, cache_seqlens=lens, causal=wl.causal,
                                                   eps=wl.eps, num_splits=splits)
        assert da.diffattn_get_device_status() == 0
        assert torch.equal(lam1, lam)
        assert torch.equal(one, two)
