"""Failure detection on the GPU without a fault: every device-side wait is
bounded.  The testing hook makes the kernels stop issuing their input copies
after a few chunks, so the next wait waits on a barrier nothing completes and
must run out after the (short) limit; the kernels must drain their own
copies, record the status word and return, the host must report
GDN_ERR_DEVICE_TIMEOUT, and the context must stay usable for a normal call
afterwards."""
import pytest
import torch

import hybrid_model_recurrent_gb300 as gdn
import synth
from parity_util import assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("algo", ["per_token", "chunked", "two_pass"])
def test_wait_limit_expiry_is_reported_and_recoverable(algo):
    gdn.build()
    w = synth.Workload("fd", [4096, 3000], 8, 128, 128, torch.bfloat16, torch.bfloat16, 0.95, 1.0, "uniform",
                       seed=91)
    inp = synth.make_inputs(w, device="cuda")
    ck = [[1024, 4096], [512]]
    ref = gdn.gdn_prefill_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, w.cu_seqlens, ckpt_pos=ck, algo=algo)
    torch.cuda.synchronize()
    nbytes = gdn.lib().gdn_workspace_size_two_pass(7096, 8, 2) if algo == "two_pass" else gdn.lib().gdn_workspace_size()
    ws = torch.zeros(int(nbytes), dtype=torch.uint8, device="cuda")
    try:
        gdn.set_wait_limit_ns(20_000_000)   # 20 ms
        gdn.debug_stall_after(3)
        gdn.gdn_prefill_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, w.cu_seqlens, ckpt_pos=ck, algo=algo, ws=ws)
        torch.cuda.synchronize()
        assert gdn.read_status(ws=ws) == gdn.GDN_ERR_DEVICE_TIMEOUT, "an unfed wait must run out and be reported"
    finally:
        gdn.debug_stall_after(-1)
        gdn.set_wait_limit_ns(0)   # back to the default
    gdn.clear_status(ws=ws)
    again = gdn.gdn_prefill_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, w.cu_seqlens, ckpt_pos=ck, algo=algo,
                                 ws=ws)
    torch.cuda.synchronize()
    assert gdn.read_status(ws=ws) == gdn.GDN_OK
    assert torch.equal(again["S_final"], ref["S_final"]) and torch.equal(again["ckpt_states"], ref["ckpt_states"])
    assert_close(again["o"].float(), ref["o"].float(), "output after recovery")
