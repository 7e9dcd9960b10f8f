"""Failure detection on the GPU without a fault: a pipeline wait that runs out.

The test hook makes the bf16 forward's copy producer issue no loads, so every
wait on the copy barriers is on a barrier nothing will complete. With a short
wait limit each CTA gives up, records DIFFATTN_ERR_TIMEOUT, frees its tensor
memory and returns; the host reads the status, and the next normal call on the
same context is correct.
"""
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
    yield
    da.diffattn_set_fault_injection(0)
    da.diffattn_set_wait_timeout_ns(0)


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
