"""The allocation-free cache forward (diffattn_fwd_kvcache_noalloc).

Its key-split scratch is the library's static device array rather than a
workspace the caller allocates, for callers that cannot allocate device memory.
Checked against the workspace entry point (diffattn_fwd_kvcache) on the same
inputs, within the bf16 tolerance of the other parity tests, on two calls in a
row with different inputs (the second call reuses the array the first one
filled), plus the rejection of shapes whose partials exceed the array.
This file is collected last so a failure here leaves every other test run.
"""
import ctypes

import pytest
import torch

import differential_attention_diffattn_gb300 as da
from differential_attention_diffattn_gb300 import _lib
from differential_attention_diffattn_gb300 import workloads as W

from gpu_util import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    da.build()
    da.load_library()
    torch.cuda.set_device(0)


def _run_both(inp):
    dev = "cuda"
    wl = inp.wl
    li = da.diffattn_lambda_init(wl.depth)
    lam = da.diffattn_lambda(inp.lambda_q1.to(dev), inp.lambda_k1.to(dev), inp.lambda_q2.to(dev),
                             inp.lambda_k2.to(dev), li)
    args = (inp.q.to(dev), inp.k_cache.to(dev), inp.v_cache.to(dev), lam, li, inp.subln_w.to(dev))
    lens = inp.cache_seqlens.to(dev)
    ref = da.diffattn_fwd_kvcache(*args, cache_seqlens=lens, causal=wl.causal, eps=wl.eps)
    got = da.diffattn_fwd_kvcache_noalloc(*args, cache_seqlens=lens, causal=wl.causal, eps=wl.eps)
    assert da.diffattn_get_device_status() == 0
    return got, ref


def test_noalloc_matches_workspace_entry_on_two_calls():
    wl = W.KvWorkload("n", num_heads=16, num_kv_heads=4, d=64, dv=128, depth=12, batch=4, q_len=1, capacity=3000)
    for seed, lens in ((61, [3000, 1500, 17, 2222]), (62, [5, 2999, 3000, 640])):
        got, ref = _run_both(W.generate_kv(wl, seed=seed, lengths=lens))
        compare(got, ref.double().cpu().numpy(), "bf16")


def test_noalloc_rejects_shapes_beyond_the_array():
    wl = W.KvWorkload("n", num_heads=16, num_kv_heads=4, d=64, dv=128, depth=12, batch=64, q_len=4,
                      capacity=8192)
    desc = _lib.kv_desc(torch.empty(64, 4, 16, 128, dtype=torch.bfloat16),
                        torch.empty(1, 8192, 4, 128, dtype=torch.bfloat16),
                        torch.empty(1, 8192, 4, 128, dtype=torch.bfloat16), num_splits=32)
    assert da.diffattn_fwd_kvcache_workspace_size(desc) > (16 << 20)
    vp = ctypes.c_void_p
    fake = vp(0x10000)  # never dereferenced: the call must fail before any launch
    st = da.load_library().diffattn_fwd_kvcache_noalloc(ctypes.byref(desc), fake, fake, fake, None, fake, 0, 0.2,
                                                        fake, 1, fake, None)
    assert st == 2  # DIFFATTN_ERR_UNSUPPORTED
    del wl


def test_noalloc_takes_fewer_splits_when_the_planned_ones_do_not_fit():
    # 50 sequences x 4 kv heads = 200 split groups: on 152 SMs (two split CTAs
    # each) the automatic plan takes 3 splits, whose partials (about 20 MB) exceed
    # the array; the allocation-free entry takes 2 instead of rejecting the shape.
    wl = W.KvWorkload("n", num_heads=16, num_kv_heads=4, d=64, dv=128, depth=12, batch=50, q_len=8,
                      capacity=1024)
    inp = W.generate_kv(wl, seed=63)
    desc = _lib.kv_desc(inp.q, inp.k_cache, inp.v_cache)
    if da.diffattn_fwd_kvcache_workspace_size(desc) <= (16 << 20):
        pytest.skip("on this device the automatic plan already fits the array")
    for _ in range(2):
        got, ref = _run_both(inp)
        compare(got, ref.double().cpu().numpy(), "bf16")


def test_noalloc_with_host_lengths():
    """The allocation-free entry with a host copy of the lengths (the split plan
    from them) against the workspace entry given the same lengths."""
    wl = W.KV_WORKLOADS["decode_b16_q4_ragged"]
    inp = W.generate_kv(wl, seed=64)
    dev = "cuda"
    li = da.diffattn_lambda_init(wl.depth)
    lam = da.diffattn_lambda(inp.lambda_q1.to(dev), inp.lambda_k1.to(dev), inp.lambda_q2.to(dev),
                             inp.lambda_k2.to(dev), li)
    args = (inp.q.to(dev), inp.k_cache.to(dev), inp.v_cache.to(dev), lam, li, inp.subln_w.to(dev))
    lens = inp.cache_seqlens.to(dev)
    host = inp.cache_seqlens.tolist()
    ref = da.diffattn_fwd_kvcache(*args, cache_seqlens=lens, causal=wl.causal, eps=wl.eps, host_seqlens=host)
    for _ in range(2):
        got = da.diffattn_fwd_kvcache_noalloc(*args, cache_seqlens=lens, causal=wl.causal, eps=wl.eps,
                                              host_seqlens=host)
        assert da.diffattn_get_device_status() == 0
        compare(got, ref.double().cpu().numpy(), "bf16")
