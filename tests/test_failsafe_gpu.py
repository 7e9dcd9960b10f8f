"""Failure detection on the GPU without a fault: a pipeline wait that runs out.

The test hook makes the bf16 forward's copy producer issue no loads, so every
wait on the copy barriers is on a barrier nothing will complete. With a short
wait limit each CTA gives up, records DIFFATTN_ERR_TIMEOUT, frees its tensor
memory and returns; the host reads the status, and the next normal call on the
same context is correct.
"""
import os

import pytest
import torch

import differential_attention_diffattn_gb300 as da
from differential_attention_diffattn_gb300 import workloads as W

from gpu_util import compare, oracle_out, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    da.build()
    da.load_library()
    torch.cuda.set_device(0)
    prev = os.environ.get("DIFFATTN_TEST_HOOKS")
    os.environ["DIFFATTN_TEST_HOOKS"] = "1"  # the library honours its test hook only with this set
    yield
    da.diffattn_set_fault_injection(0)
    da.diffattn_set_wait_timeout_ns(0)
    if prev is None:
        del os.environ["DIFFATTN_TEST_HOOKS"]
    else:
        os.environ["DIFFATTN_TEST_HOOKS"] = prev


# packed: the one-item-per-CTA kernel; an unpacked batch of 3 x 1000 tokens
# (384 items): the persistent kernel, whose warps must all leave their loops
@pytest.mark.parametrize("lens,packed", [([256, 100], True), ([1000, 1000, 1000], False)])
def test_wait_timeout_reported_and_context_usable(lens, packed):
    inp = W.generate(W.WORKLOADS["b2_t512_gqa"], seed=71, seq_lens=lens)
    da.diffattn_set_wait_timeout_ns(20_000_000)  # 20 ms
    da.diffattn_set_fault_injection(1)
    try:
        with pytest.raises(AssertionError, match="timed out"):
            run_gpu(inp, packed=packed)
    finally:
        da.diffattn_set_fault_injection(0)
        da.diffattn_set_wait_timeout_ns(0)
    assert da.diffattn_get_device_status() == 0  # the read cleared it
    compare(run_gpu(inp, packed=packed), oracle_out(inp), "bf16")


def test_epilogue_held_back_changes_nothing():
    """The persistent kernel's epilogue warpgroup paused ~20 us before each item,
    so that the softmax warps run ahead of it, also through items of one key
    tile (which need no P V before their scores): the same bits, no timeout.
    With one 1/l barrier for all items instead of one per item parity, its phase
    could run two ahead of the epilogue here and the epilogue's wait ran out."""
    lens = [1000, 90, 700, 128, 40, 1000, 300, 129, 64, 900, 1, 500, 256, 77, 1000, 640]
    inp = W.generate(W.WORKLOADS["b2_t512_gqa"], seed=72, seq_lens=lens)
    t = {k: v.cuda() for k, v in (("q", inp.q), ("k", inp.k), ("v", inp.v))}
    lam = torch.ones(1, dtype=torch.float32, device="cuda")
    assert da.diffattn_fwd_kernel(t["q"], t["k"], t["v"], lam, inp.subln_w.cuda(), cu_seqlens=inp.cu_seqlens.cuda(),
                                  max_seqlen=max(lens)) == "diffattn_fwd_bf16_persistent_kernel"
    ref = run_gpu(inp)
    da.diffattn_set_wait_timeout_ns(200_000_000)  # 200 ms
    da.diffattn_set_fault_injection(2)
    try:
        got = run_gpu(inp)  # asserts a zero status word
    finally:
        da.diffattn_set_fault_injection(0)
        da.diffattn_set_wait_timeout_ns(0)
    assert torch.equal(got, ref)
