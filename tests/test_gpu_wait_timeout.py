"""The failure path of the kernels' bounded waits, without a GPU fault: a
wait that nothing satisfies gives up after its cycle limit, the status word
reports MOE_ERR_TIMEOUT, and the same context then runs the layer correctly."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, built, get_config, gpu_forward, make, oracle_full, ws_status

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return built()


def test_bounded_wait_times_out_and_context_stays_usable():
    import time
    import bit_block_scaled_gb300 as moe
    ws = ws_status()
    t0 = time.time()
    moe.moe_wait_selftest(ws)
    st = moe.moe_read_status(ws)          # synchronises
    elapsed = time.time() - t0
    assert st == 4, moe.moe_status_string(st)
    assert 0.2 < elapsed < 30.0           # about a second of cycles, then it returns
    moe.moe_clear_status(ws)
    assert moe.moe_read_status(ws) == 0
    cfg = get_config("c0")
    L, N = make(cfg)
    out, ws2 = gpu_forward(L, cfg)
    assert moe.moe_read_status(ws2) == 0
    assert_close(out.float().cpu().numpy(), oracle_full(N, cfg)["out"], "forward after a time-out")
