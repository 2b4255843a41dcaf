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


@pytest.mark.parametrize("kind", ["paged", "fp8", "paged_fp8"])
@pytest.mark.parametrize("variant", [1, 2])
def test_withheld_q_times_out_in_paged_and_fp8_kernels(cuda_device, kind, variant):
    """The same failure path in the paged and FP8-QK^T instantiations: their extra
    waits (the key-scale ring) and copies (page pieces, bulk scale copies) give up
    and drain as well, and the context stays usable."""
    import gqa_chunked_prefill_gb300 as gqa
    from gqa_inputs import make_paged_batch, make_varlen
    assert gqa.gqa_prefill_poll() == 0
    q, k, v, cu_q, cu_k = make_varlen([(100, 900)], 9)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.zeros_like(qd)
    lse = torch.zeros(100, 24, device=dev)
    force = dict(wait_timeout_us=50_000, test_withhold_q=True, force_variant=variant)
    if kind == "paged":
        kc, vc, table, kv_lens = make_paged_batch(k, v, cu_k, 16, seed=10)
        gqa.gqa_prefill_attn_paged_varlen_ex(qd, kc.to(dev), vc.to(dev), table.to(dev),
                                             table.shape[1], kc.shape[0], 16, out, lse, cu_q,
                                             kv_lens, 24, 4, 256, 1 / 16, **force)
    else:
        q8 = torch.empty(qd.shape, dtype=torch.uint8, device=dev)
        qs = torch.empty((100, 24), dtype=torch.float32, device=dev)
        gqa.gqa_quantize_q_fp8(qd, q8, qs, 100, 24, 256)
        if kind == "fp8":
            k8 = torch.empty(kd.shape, dtype=torch.uint8, device=dev)
            ks = torch.empty((4, 900), dtype=torch.float32, device=dev)
            gqa.gqa_quantize_k_fp8(kd, k8, ks, 900, 4, 256, 900)
            gqa.gqa_prefill_attn_fp8qk_ex(q8, qs, k8, ks, 900, vd, out, lse, 100, 900, 24, 4, 256,
                                          1 / 16, **force)
        else:
            kc, vc, table, kv_lens = make_paged_batch(k, v, cu_k, 48, seed=11)
            rows = kc.shape[0] * 48
            kc8 = torch.empty(kc.shape, dtype=torch.uint8, device=dev)
            kcs = torch.empty((4, rows), dtype=torch.float32, device=dev)
            gqa.gqa_quantize_k_fp8(kc.to(dev), kc8, kcs, rows, 4, 256, rows)
            gqa.gqa_prefill_attn_paged_fp8qk_varlen_ex(q8, qs, kc8, kcs, rows, vc.to(dev),
                                                       table.to(dev), table.shape[1], kc.shape[0],
                                                       48, out, lse, cu_q, kv_lens, 24, 4, 256,
                                                       1 / 16, **force)
    assert gqa.gqa_prefill_poll() == gqa.GqaStatus.ERR_DEVICE_TIMEOUT
    assert gqa.gqa_prefill_poll() == 0
    o2, l2, _ = run_gpu(q, k, v, 1 / 16)
    ref_o, ref_l = oracle.attention(q, k, v, 1 / 16)
    check_close(o2.double().cpu().numpy(), l2.double().cpu().numpy(), ref_o, ref_l,
                f"after {kind} timeout")
