"""Failure detection on the GPU without a fault: the producer withholds the first
Q tile of every CTA (a test-only option), so each consumer wait runs out after a
short limit. The kernel must record GQA_ERR_DEVICE_TIMEOUT in the device status
word, drain its TMA copies, free tensor memory and return, leaving the context
usable: the next normal call on the same stream must succeed and be correct."""
import pytest
import torch

import oracle
from gqa_inputs import make_qkv
from tests.gpu_helpers import check_close, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", [1, 2])
def test_withheld_q_times_out_and_context_survives(cuda_device, variant):
    """variant 2 also covers a CTA pair giving up together (leader and peer)."""
    import gqa_chunked_prefill_gb300 as gqa
    assert gqa.gqa_prefill_poll() == 0
    q, k, v = make_qkv(100, 900, seed=5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.zeros_like(qd)
    lse = torch.zeros(100, 24, device="cuda")
    rc, plan = gqa.gqa_prefill_attn_ex(qd, kd, vd, out, lse, 100, 900, 24, 4, 256, 1 / 16,
                                       wait_timeout_us=50_000, test_withhold_q=True,
                                       force_variant=variant)
    assert rc == 0 and plan["variant"] == variant  # launched; the device reports the failure
    status = gqa.gqa_prefill_poll()
    assert status == gqa.GqaStatus.ERR_DEVICE_TIMEOUT
    assert gqa.gqa_prefill_poll() == 0  # polling clears the word
    # the context is still usable and the next call is exact
    o2, l2, _ = run_gpu(q, k, v, 1 / 16)
    ref_o, ref_l = oracle.attention(q, k, v, 1 / 16)
    check_close(o2.double().cpu().numpy(), l2.double().cpu().numpy(), ref_o, ref_l, "after timeout")
