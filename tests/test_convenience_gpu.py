"""The convenience wrappers of the package (output allocation and argument
marshalling only) give exactly what the entry points they wrap give."""
import pytest
import torch

from gqa_inputs import make_paged_batch, make_qkv, make_varlen

pytestmark = pytest.mark.gpu
SCALE = 1.0 / 16.0


def test_wrappers_match_entry_points(cuda_device):
    import gqa_chunked_prefill_gb300 as gqa
    lens = [(43, 300), (1, 2000), (129, 1001)]
    q, k, v, cu_q, cu_k = (x.cuda() if hasattr(x, "cuda") else x for x in make_varlen(lens, 77))
    o1, l1 = gqa.attention_varlen(q, k, v, cu_q, cu_k, SCALE)
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    gqa.gqa_prefill_attn_varlen(q, k, v, o2, l2, cu_q, cu_k, 24, 4, 256, SCALE)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)

    kc, vc, table, kv_lens = make_paged_batch(k.cpu(), v.cpu(), cu_k, 784, seed=78)
    kc, vc, table = kc.cuda(), vc.cuda(), table.cuda()
    o3, l3 = gqa.attention_paged(q, kc, vc, table, kv_lens, cu_q, SCALE)
    o3e = torch.empty_like(q)
    l3e = torch.empty_like(l1)
    _, plan_p = gqa.gqa_prefill_attn_paged_varlen_ex(q, kc, vc, table, table.shape[1], kc.shape[0],
                                                     784, o3e, l3e, cu_q, kv_lens, 24, 4, 256, SCALE)
    assert torch.equal(o3, o3e) and torch.equal(l3, l3e)
    # Paged calls may prefer the CTA pair where dense ones do not: the dense batch
    # with the paged plan's variant gives the same bits.
    o3d = torch.empty_like(q)
    l3d = torch.empty_like(l1)
    gqa.gqa_prefill_attn_varlen_ex(q, k, v, o3d, l3d, cu_q, cu_k, 24, 4, 256, SCALE,
                                   force_variant=plan_p["variant"])
    assert torch.equal(o3, o3d) and torch.equal(l3, l3d)

    q8, qs = gqa.quantize_fp8(q)
    k8, ks = gqa.quantize_fp8(k, cu_k)
    o4, l4 = gqa.attention_fp8qk(q8, qs, k8, ks, v, cu_q, cu_k, SCALE)
    o5 = torch.empty_like(q)
    l5 = torch.empty_like(l1)
    gqa.gqa_prefill_attn_fp8qk_varlen_ex(q8, qs, k8, ks, ks.shape[1], v, o5, l5, cu_q, cu_k, 24, 4,
                                         256, SCALE)
    assert torch.equal(o4, o5) and torch.equal(l4, l5)

    qs1, ks1, vs1 = (t.cuda() for t in make_qkv(50, 400, seed=79))
    o6, l6 = gqa.attention(qs1, ks1, vs1, SCALE)
    o6e = torch.empty_like(qs1)
    l6e = torch.empty_like(l6)
    gqa.gqa_prefill_attn(qs1, ks1, vs1, o6e, l6e, 50, 400, 24, 4, 256, SCALE)
    assert torch.equal(o6, o6e) and torch.equal(l6, l6e)
    tbl = torch.arange(1, dtype=torch.int32, device="cuda")
    kc1, vc1 = ks1.reshape(1, 400, 4, 256), vs1.reshape(1, 400, 4, 256)
    o7, l7 = gqa.attention_paged(qs1, kc1, vc1, tbl, 400, scale=SCALE)
    o7e = torch.empty_like(qs1)
    l7e = torch.empty_like(l6)
    _, plan7 = gqa.gqa_prefill_attn_paged_ex(qs1, kc1, vc1, tbl, 1, 400, o7e, l7e, 50, 400, 24, 4,
                                             256, SCALE)
    o6d = torch.empty_like(qs1)
    l6d = torch.empty_like(l6)
    gqa.gqa_prefill_attn_ex(qs1, ks1, vs1, o6d, l6d, 50, 400, 24, 4, 256, SCALE,
                            force_variant=plan7["variant"])
    torch.cuda.synchronize()
    assert gqa.gqa_prefill_poll() == 0
    assert torch.equal(o7, o7e) and torch.equal(l7, l7e)
    assert torch.equal(o7, o6d) and torch.equal(l7, l6d)
