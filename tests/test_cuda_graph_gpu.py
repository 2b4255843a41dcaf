"""The entry points are stream-ordered throughout (planning and tensor maps on
the host, split partials from a stream-ordered pool, programmatic dependent
launches), so a call can be captured into a CUDA graph once and replayed: the
graph holds the plan, the tensor maps and the pointers, and each replay reads
whatever the input buffers hold then. Checks: a replay equals the direct call
bit for bit, and after new values are written into the same input buffers a
replay equals a direct call on those values."""
import pytest
import torch

from gqa_inputs import make_paged_batch, make_qkv, make_varlen

pytestmark = pytest.mark.gpu
SCALE = 1.0 / 16.0


def capture(fn, stream):
    """fn(stream) once for warm-up (library set-up happens outside the capture), then
    captured into a graph."""
    fn(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn(stream)
    torch.cuda.synchronize()
    return g


def check_replay(fn, inputs, outputs, new_inputs, stream):
    import gqa_chunked_prefill_gb300 as gqa
    g = capture(fn, stream)
    fn(stream)
    torch.cuda.synchronize()
    direct = [o.clone() for o in outputs]
    for o in outputs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(o, d) for o, d in zip(outputs, direct))
    for buf, new in zip(inputs, new_inputs):
        buf.copy_(new)
    g.replay()
    torch.cuda.synchronize()
    replayed = [o.clone() for o in outputs]
    fn(stream)
    torch.cuda.synchronize()
    assert all(torch.equal(o, r) for o, r in zip(outputs, replayed))
    assert not torch.equal(replayed[0], direct[0])
    assert gqa.gqa_prefill_poll() == 0


@pytest.mark.parametrize("q_len,kv_len,splits", [(300, 1000, 3), (1, 4096, 16), (129, 129, 1),
                                                 (300, 1000, -1), (1, 4096, -1)])
def test_dense_call_in_a_graph(cuda_device, q_len, kv_len, splits):
    import gqa_chunked_prefill_gb300 as gqa
    s = torch.cuda.Stream()
    q, k, v = (t.cuda() for t in make_qkv(q_len, kv_len, seed=1))
    q2, k2, v2 = (t.cuda() for t in make_qkv(q_len, kv_len, seed=2))
    out = torch.empty_like(q)
    lse = torch.empty((q_len, 24), dtype=torch.float32, device="cuda")

    def fn(stream):
        gqa.gqa_prefill_attn_ex(q, k, v, out, lse, q_len, kv_len, 24, 4, 256, SCALE,
                                stream=stream, force_splits=splits)

    check_replay(fn, [q, k, v], [out, lse], [q2, k2, v2], s)


def test_batched_paged_call_in_a_graph(cuda_device):
    import gqa_chunked_prefill_gb300 as gqa
    s = torch.cuda.Stream()
    lens = [(43, 300), (1, 2000), (129, 1000)]
    q, k, v, cu_q, cu_k = make_varlen(lens, 3)
    q2, _, _, _, _ = make_varlen(lens, 4)
    kc, vc, table, kv_lens = make_paged_batch(k, v, cu_k, 48, seed=5)
    qd, kcd, vcd, td = q.cuda(), kc.cuda(), vc.cuda(), table.cuda()
    out = torch.empty_like(qd)
    lse = torch.empty((qd.shape[0], 24), dtype=torch.float32, device="cuda")

    def fn(stream):
        gqa.gqa_prefill_attn_paged_varlen_ex(qd, kcd, vcd, td, table.shape[1], kc.shape[0], 48,
                                             out, lse, cu_q, kv_lens, 24, 4, 256, SCALE,
                                             stream=stream, force_splits=2)

    check_replay(fn, [qd], [out, lse], [q2.cuda()], s)


def test_fp8qk_call_in_a_graph(cuda_device):
    import gqa_chunked_prefill_gb300 as gqa
    s = torch.cuda.Stream()
    q, k, v = (t.cuda() for t in make_qkv(200, 1500, seed=6))
    q2 = make_qkv(200, 1500, seed=7)[0].cuda()
    q8 = torch.empty(q.shape, dtype=torch.uint8, device="cuda")
    qs = torch.empty((200, 24), dtype=torch.float32, device="cuda")
    k8 = torch.empty(k.shape, dtype=torch.uint8, device="cuda")
    ks = torch.empty((4, 1500), dtype=torch.float32, device="cuda")
    gqa.gqa_quantize_k_fp8(k, k8, ks, 1500, 4, 256, 1500)
    out = torch.empty_like(q)
    lse = torch.empty((200, 24), dtype=torch.float32, device="cuda")

    def fn(stream):  # the per-chunk Q quantisation is part of the captured step
        gqa.gqa_quantize_q_fp8(q, q8, qs, 200, 24, 256, stream=stream)
        gqa.gqa_prefill_attn_fp8qk_ex(q8, qs, k8, ks, 1500, v, out, lse, 200, 1500, 24, 4, 256,
                                      SCALE, stream=stream, force_splits=3)

    check_replay(fn, [q], [out, lse], [q2], s)
