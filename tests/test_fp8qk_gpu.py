"""GPU parity of the quantised-QK^T path (E4M3 codes, per-vector scales).

1. The quantise kernels give the oracle's codes and scales bit for bit (both
   sides take every rounding decision in FP32: s = amax / 448, code = E4M3(x / s)).
2. gqa_prefill_attn_fp8qk matches the FP64 oracle run on the dequantised query
   and keys (the oracle quantises the same BF16 inputs itself) at the
   acceptance tolerance of the BF16 path: products of E4M3 codes are exact in
   FP32, and the scales are restored in FP32 before the softmax, so what is left
   is the BF16 rounding of P and of the output, as in the BF16 path.
3. The quantisation error itself (against unquantised attention) is reported by
   a loose bound, not a parity claim.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_inputs import WORKLOADS, make_qkv, make_workload, sample_rows
from tests.gpu_helpers import check_close, gather_rows, item_cover_rows, unchecked_items

pytestmark = pytest.mark.gpu
SCALE = 1.0 / 16.0


def quantize_gpu(q, k):
    """GPU codes/scales: q_fp8 [q_len,24,256] u8, q_scale [q_len,24], k_fp8 [kv_len,4,256] u8,
    k_scale [4, stride] (head-major, stride = kv_len rounded up to 4)."""
    import gqa_chunked_prefill_gb300 as gqa
    dev = torch.device("cuda:0")
    qd, kd = q.to(dev).contiguous(), k.to(dev).contiguous()
    q_len, kv_len = qd.shape[0], kd.shape[0]
    stride = max(4, -(-kv_len // 4) * 4)
    q8 = torch.empty(qd.shape, dtype=torch.uint8, device=dev)
    qs = torch.empty((q_len, 24), dtype=torch.float32, device=dev)
    k8 = torch.empty(kd.shape, dtype=torch.uint8, device=dev)
    ks = torch.full((4, stride), float("nan"), dtype=torch.float32, device=dev)
    gqa.gqa_quantize_q_fp8(qd, q8, qs, q_len, 24, 256)
    gqa.gqa_quantize_k_fp8(kd, k8, ks, kv_len, 4, 256, stride)
    torch.cuda.synchronize()
    return q8, qs, k8, ks, stride


def run_fp8(q, k, v, scale, **force):
    import gqa_chunked_prefill_gb300 as gqa
    dev = torch.device("cuda:0")
    q8, qs, k8, ks, stride = quantize_gpu(q, k)
    vd = v.to(dev).contiguous()
    q_len, kv_len = q.shape[0], k.shape[0]
    out = torch.empty((q_len, 24, 256), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((q_len, 24), dtype=torch.float32, device=dev)
    _, plan = gqa.gqa_prefill_attn_fp8qk_ex(q8, qs, k8, ks, stride, vd, out, lse, q_len, kv_len,
                                            24, 4, 256, scale, **force)
    torch.cuda.synchronize()
    assert gqa.gqa_prefill_poll() == 0
    return out, lse, plan


def oracle_fp8(q, k, v, scale, rows=None):
    qc, qs = oracle.quantize_e4m3(q)
    kc, ks = oracle.quantize_e4m3(k)
    return oracle.fp8qk_attention(qc, qs, kc, ks, v, scale, rows=rows)


@pytest.mark.parametrize("q_len,kv_len", [(1, 1), (43, 300), (300, 1000), (7, 4097)])
def test_quantize_kernels_match_oracle_bit_for_bit(cuda_device, q_len, kv_len):
    q, k, _ = make_qkv(q_len, kv_len, seed=q_len + 7 * kv_len)
    q = q.clone()
    k = k.clone()
    q[0, 3] = 0                                  # an all-zero vector: s = 0, codes 0
    k[-1, 2] = 0
    k[0, 1] = k[0, 1] * 1e-30                    # scale far below 1: tiny but normal
    q[-1, 0, :128] = q[-1, 0, :128] * 1e-6       # half the vector in E4M3's subnormal range
    q8, qs, k8, ks, _ = quantize_gpu(q, k)
    qc, qsc = oracle.quantize_e4m3(q)
    kc, ksc = oracle.quantize_e4m3(k)
    assert np.array_equal(q8.cpu().numpy(), qc) and np.array_equal(qs.cpu().numpy(), qsc)
    assert np.array_equal(k8.cpu().numpy(), kc)
    assert np.array_equal(ks[:, :kv_len].cpu().numpy(), ksc.T)


def _e4m3_boundary_vectors(rows, heads, seed):
    """Vectors whose quotients x / s sit on or next to E4M3 rounding boundaries: each
    holds 448 (so amax = 448 and s = 1 exactly: x / s = x) and otherwise values at the
    midpoints between neighbouring E4M3 numbers (ties, rounded to even), one BF16 step
    either side of them, the boundary of E4M3's subnormal range and the halfway point
    below its least code; then the same vectors scaled by 2^k and by 3 (s no longer a
    power of two: quotients land next to the boundaries instead of on them)."""
    g = torch.Generator().manual_seed(seed)
    vals = []
    for e in range(-6, 9):                      # normal E4M3: midpoints (1 + (2m+1)/16) 2^e
        for m in range(8):
            vals.append((1 + (2 * m + 1) / 16) * 2.0 ** e)
    for m in range(8):                          # subnormal E4M3: midpoints (2m+1) 2^-10
        vals.append((2 * m + 1) * 2.0 ** -10)
    vals += [2.0 ** -6, 2.0 ** -10, 2.0 ** -11, 448.0, 464.0]
    base = torch.tensor(vals, dtype=torch.float32)
    near = torch.cat([base, torch.nextafter(base.bfloat16().float(), torch.tensor(0.0)),
                      torch.nextafter(base.bfloat16().float(), torch.tensor(1e9))])
    x = torch.empty(rows, heads, 256)
    for r in range(rows):
        for h in range(heads):
            idx = torch.randint(0, near.numel(), (255,), generator=g)
            sign = torch.where(torch.rand(255, generator=g) < 0.5, -1.0, 1.0)
            x[r, h, 0] = 448.0
            x[r, h, 1:] = near[idx] * sign
    scaled = [x, x * 2.0 ** -5, x * 2.0 ** 7, x * 3.0, x / 3.0]
    return torch.cat(scaled).clamp(-3e38, 3e38).to(torch.bfloat16)


def test_quantize_codes_at_e4m3_rounding_boundaries(cuda_device):
    """The kernels divide each value by its vector's scale with an IEEE
    round-to-nearest division, then round to E4M3: on inputs built around E4M3
    rounding boundaries (midpoints between codes, their BF16 neighbours, the
    subnormal range, saturation) the codes and scales must equal the oracle's bit
    for bit."""
    q = _e4m3_boundary_vectors(8, 24, seed=91)
    k = _e4m3_boundary_vectors(8, 4, seed=92)
    q8, qs, k8, ks, _ = quantize_gpu(q, k)
    qc, qsc = oracle.quantize_e4m3(q)
    kc, ksc = oracle.quantize_e4m3(k)
    assert np.array_equal(q8.cpu().numpy(), qc) and np.array_equal(qs.cpu().numpy(), qsc)
    assert np.array_equal(k8.cpu().numpy(), kc)
    assert np.array_equal(ks[:, :k.shape[0]].cpu().numpy(), ksc.T)


@pytest.mark.parametrize("q_len,kv_len", [(1, 1), (5, 300), (43, 300), (100, 100), (129, 1000),
                                          (22, 2000)])
@pytest.mark.parametrize("variant", [1, 2])
def test_fp8qk_small_shapes_every_element(cuda_device, q_len, kv_len, variant):
    q, k, v = make_qkv(q_len, kv_len, seed=5 * q_len + kv_len)
    out, lse, plan = run_fp8(q, k, v, SCALE, force_variant=variant)
    assert plan["variant"] == variant
    ref_o, ref_l = oracle_fp8(q, k, v, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                f"fp8 {q_len}x{kv_len}")


@pytest.mark.parametrize("splits,grid,variant", [(3, 0, 1), (3, 5, 1), (2, 0, 2), (3, 6, 2),
                                                 (32, 0, 1), (-1, 0, 1), (-1, 6, 2)])
def test_fp8qk_split_tail_every_element(cuda_device, splits, grid, variant):
    q, k, v = make_qkv(129, 1000, seed=31)
    out, lse, _ = run_fp8(q, k, v, SCALE, force_splits=splits, force_grid=grid,
                          force_variant=variant)
    ref_o, ref_l = oracle_fp8(q, k, v, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                f"fp8 split {splits} grid {grid}")


@pytest.mark.parametrize("name", ["q4096_kv32768", "q512_kv4096_kbias", "q3072_kv16384"])
@pytest.mark.parametrize("variant", [0, 1])
def test_fp8qk_workload_full_size(cuda_device, name, variant):
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    out, lse, plan = run_fp8(q, k, v, w.scale, force_variant=variant)
    rows = item_cover_rows(w.q_len, w.n_q_heads, sample_rows(w.q_len, w.n_q_heads, 1200, seed=12))
    assert unchecked_items(rows, w.q_len, 21 * plan["variant"]) == []
    ref_o, ref_l = oracle_fp8(q, k, v, w.scale, rows=rows)
    got_o, got_l = gather_rows(out, lse, rows)
    check_close(got_o, got_l, ref_o, ref_l, f"fp8 {name}")


def test_fp8qk_quantisation_error_is_small_against_bf16_attention(cuda_device):
    """Not parity: the method's own error. With N(0,1) data the E4M3 codes (3
    mantissa bits, relative step 2^-3) perturb each score by about
    2^-4 * scale * |q| |k| / sqrt(d); outputs stay within a few 1e-2."""
    q, k, v = make_qkv(64, 2000, seed=77)
    out, lse, _ = run_fp8(q, k, v, SCALE)
    ref_o, ref_l = oracle.attention(q, k, v, SCALE)
    err = np.abs(out.double().cpu().numpy() - ref_o)
    assert err.mean() < 5e-3 and err.max() < 6e-2
    assert np.abs(lse.double().cpu().numpy() - ref_l).max() < 5e-2


# --- quantised QK^T in batched calls, dense and paged -----------------------------

def _fp8_batch_inputs(lens, seed):
    from gqa_inputs import make_varlen
    return make_varlen(lens, seed)


def quantize_batch_gpu(q, k, cu_k):
    """GPU codes/scales of a packed batch; key scales in the batched layout (each
    sequence from a column that is a multiple of 4)."""
    import gqa_chunked_prefill_gb300 as gqa
    dev = torch.device("cuda:0")
    qd, kd = q.to(dev).contiguous(), k.to(dev).contiguous()
    starts, cols = gqa.key_scale_columns(cu_k)
    stride = max(4, cols)
    q8 = torch.empty(qd.shape, dtype=torch.uint8, device=dev)
    qs = torch.empty((qd.shape[0], 24), dtype=torch.float32, device=dev)
    k8 = torch.empty(kd.shape, dtype=torch.uint8, device=dev)
    ks = torch.full((4, stride), float("nan"), dtype=torch.float32, device=dev)
    gqa.gqa_quantize_q_fp8(qd, q8, qs, qd.shape[0], 24, 256)
    gqa.gqa_quantize_k_fp8_varlen(kd, k8, ks, cu_k, 4, 256, stride)
    torch.cuda.synchronize()
    return q8, qs, k8, ks, stride, starts


def test_batched_key_scales_land_in_their_columns(cuda_device):
    q, k, v, cu_q, cu_k = _fp8_batch_inputs([(3, 5), (2, 7), (0, 1), (4, 9)], 800)
    _, _, k8, ks, _, starts = quantize_batch_gpu(q, k, cu_k)
    kc, ksc = oracle.quantize_e4m3(k)
    assert np.array_equal(k8.cpu().numpy(), kc)
    for b in range(4):
        n = cu_k[b + 1] - cu_k[b]
        got = ks[:, starts[b]:starts[b] + n].cpu().numpy()
        assert np.array_equal(got, ksc[cu_k[b]:cu_k[b + 1]].T), f"sequence {b}"
    assert starts == [0, 8, 16, 20]


@pytest.mark.parametrize("variant", [1, 2])
def test_fp8qk_varlen_every_element(cuda_device, variant):
    import gqa_chunked_prefill_gb300 as gqa
    q, k, v, cu_q, cu_k = _fp8_batch_inputs([(43, 300), (1, 2000), (0, 9), (129, 1001), (2, 3)],
                                            810)
    q8, qs, k8, ks, stride, _ = quantize_batch_gpu(q, k, cu_k)
    dev = torch.device("cuda:0")
    out = torch.empty((q.shape[0], 24, 256), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((q.shape[0], 24), dtype=torch.float32, device=dev)
    gqa.gqa_prefill_attn_fp8qk_varlen_ex(q8, qs, k8, ks, stride, v.to(dev), out, lse, cu_q, cu_k,
                                         24, 4, 256, SCALE, force_variant=variant)
    torch.cuda.synchronize()
    assert gqa.gqa_prefill_poll() == 0
    qc, qsc = oracle.quantize_e4m3(q)
    kc, ksc = oracle.quantize_e4m3(k)
    ref_o, ref_l = oracle.varlen_attention(oracle.dequantize_e4m3(qc, qsc),
                                           oracle.dequantize_e4m3(kc, ksc), v, cu_q, cu_k, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l, "fp8 varlen")


@pytest.mark.parametrize("page_size", [16, 784])
@pytest.mark.parametrize("variant", [1, 2])
def test_paged_fp8qk_varlen_matches_dense(cuda_device, page_size, variant):
    """The paged FP8 batch (K codes and scales quantised in place over the whole
    cache, unused slots NaN) equals the dense FP8 batch bit for bit."""
    import gqa_chunked_prefill_gb300 as gqa
    from gqa_inputs import make_paged_batch
    q, k, v, cu_q, cu_k = _fp8_batch_inputs([(43, 300), (1, 2000), (0, 9), (129, 1000), (5, 5)], 820)
    kc, vc, table, kv_lens = make_paged_batch(k, v, cu_k, page_size, seed=821)
    dev = torch.device("cuda:0")
    rows = kc.shape[0] * page_size
    stride = -(-rows // 4) * 4
    kc8 = torch.empty(kc.shape, dtype=torch.uint8, device=dev)
    kcs = torch.empty((4, stride), dtype=torch.float32, device=dev)
    gqa.gqa_quantize_k_fp8(kc.to(dev), kc8, kcs, rows, 4, 256, stride)
    q8, qs, k8, ks, dstride, _ = quantize_batch_gpu(q, k, cu_k)
    out_p = torch.empty((q.shape[0], 24, 256), dtype=torch.bfloat16, device=dev)
    lse_p = torch.empty((q.shape[0], 24), dtype=torch.float32, device=dev)
    _, plan_p = gqa.gqa_prefill_attn_paged_fp8qk_varlen_ex(
        q8, qs, kc8, kcs, stride, vc.to(dev), table.to(dev), table.shape[1], kc.shape[0],
        page_size, out_p, lse_p, cu_q, kv_lens, 24, 4, 256, SCALE, force_variant=variant)
    out_d = torch.empty_like(out_p)
    lse_d = torch.empty_like(lse_p)
    _, plan_d = gqa.gqa_prefill_attn_fp8qk_varlen_ex(q8, qs, k8, ks, dstride, v.to(dev), out_d,
                                                     lse_d, cu_q, cu_k, 24, 4, 256, SCALE,
                                                     force_variant=variant)
    torch.cuda.synchronize()
    assert gqa.gqa_prefill_poll() == 0
    assert plan_p == plan_d
    assert torch.equal(out_p, out_d) and torch.equal(lse_p, lse_d)


@pytest.mark.parametrize("variant", [1, 2])
def test_fp8qk_zero_query_gives_the_mean_of_visible_v(cuda_device, variant):
    """A query of zeros quantises to scale 0 and codes 0: all its scores are 0, so
    its output is the mean of the visible V rows and its LSE ln(visible keys). (Its
    masked keys must stay at -inf: a zero factor must not turn them into NaN.)"""
    q, k, v = make_qkv(30, 500, seed=43)
    q[::3] = 0
    out, lse, _ = run_fp8(q, k, v, SCALE, force_variant=variant)
    ref_o, ref_l = oracle_fp8(q, k, v, SCALE)
    check_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                "fp8 zero query")
    vv = v.double().numpy()
    for t in (0, 3, 27):
        want = np.repeat(vv[:470 + t + 1].mean(axis=0), 6, axis=0)
        assert np.allclose(out[t].double().cpu().numpy(), want, rtol=2 ** -8, atol=1e-4)
        assert np.allclose(lse[t].cpu().numpy(), np.log(470 + t + 1), atol=1e-5)
