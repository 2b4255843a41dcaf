"""GPU parity of the quantised-PV path (gqa_quantize_v_fp8, gqa_prefill_attn_fp8qkpv).

Reading (the INT8 QK MMAC page, §6, names an 8-bit PV in the final submission
without its scaling): V gets one E4M3 scale per (KV head, channel) over the
call's keys; P is rounded to E4M3 as the MMA operand; the normaliser keeps the
FP32 probabilities. The oracle is attention of the dequantised Q, K and V with
exact probabilities (oracle.fp8pv_attention). What rounding P may change is
bounded per element by oracle.fp8pv_p_bound; the parity test allows that bound,
plus BF16 output rounding (2^-8 relative covers it) and 1e-4 absolute. The V
codes and scales are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_inputs import WORKLOADS, make_qkv, make_workload, sample_rows
from tests.gpu_helpers import LSE_TOL, gather_rows, item_cover_rows, unchecked_items

pytestmark = pytest.mark.gpu
SCALE = 1.0 / 16.0


def quantize_all_gpu(q, k, v):
    import gqa_chunked_prefill_gb300 as gqa
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev).contiguous() for t in (q, k, v))
    q_len, kv_len = qd.shape[0], kd.shape[0]
    kstride = max(4, -(-kv_len // 4) * 4)
    vstride = max(16, -(-kv_len // 16) * 16)
    q8 = torch.empty(qd.shape, dtype=torch.uint8, device=dev)
    qs = torch.empty((q_len, 24), dtype=torch.float32, device=dev)
    k8 = torch.empty(kd.shape, dtype=torch.uint8, device=dev)
    ks = torch.empty((4, kstride), dtype=torch.float32, device=dev)
    v8 = torch.full((4, 256, vstride), 0x7F, dtype=torch.uint8, device=dev)  # NaN codes past kv_len
    vs = torch.empty((4, 256), dtype=torch.float32, device=dev)
    gqa.gqa_quantize_q_fp8(qd, q8, qs, q_len, 24, 256)
    gqa.gqa_quantize_k_fp8(kd, k8, ks, kv_len, 4, 256, kstride)
    gqa.gqa_quantize_v_fp8(vd, v8, vs, kv_len, 4, 256, vstride)
    torch.cuda.synchronize()
    return q8, qs, k8, ks, kstride, v8, vs, vstride


def run_fp8pv(q, k, v, scale, **force):
    import gqa_chunked_prefill_gb300 as gqa
    dev = torch.device("cuda:0")
    q8, qs, k8, ks, kstride, v8, vs, vstride = quantize_all_gpu(q, k, v)
    q_len, kv_len = q.shape[0], k.shape[0]
    out = torch.empty((q_len, 24, 256), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((q_len, 24), dtype=torch.float32, device=dev)
    _, plan = gqa.gqa_prefill_attn_fp8qkpv_ex(q8, qs, k8, ks, kstride, v8, vs, vstride, out, lse,
                                              q_len, kv_len, 24, 4, 256, scale, **force)
    torch.cuda.synchronize()
    assert gqa.gqa_prefill_poll() == 0
    return out, lse, plan


def oracle_fp8pv(q, k, v, scale, rows=None):
    qc, qs = oracle.quantize_e4m3(q)
    kc, ks = oracle.quantize_e4m3(k)
    vc, vs = oracle.quantize_v_e4m3(v)
    ref_o, ref_l = oracle.fp8pv_attention(qc, qs, kc, ks, vc, vs, scale, rows=rows)
    bound = oracle.fp8pv_p_bound(oracle.dequantize_e4m3(qc, qs), oracle.dequantize_e4m3(kc, ks),
                                 oracle.dequantize_v_e4m3(vc, vs), scale, rows=rows)
    return ref_o, ref_l, bound


def check_pv(out, lse, ref_o, ref_l, bound, what):
    err = np.abs(out - ref_o)
    tol = bound + 2.0 ** -8 * np.abs(ref_o) + 1e-4
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert np.all(err <= tol), (f"{what}: error {err[worst]:.3e} above its bound {tol[worst]:.3e} "
                                f"at {worst}")
    assert np.abs(lse - ref_l).max() <= LSE_TOL, f"{what}: LSE max err {np.abs(lse - ref_l).max():.3e}"
    return err


@pytest.mark.parametrize("kv_len", [1, 37, 300, 513, 2048, 4097])
def test_quantize_v_matches_oracle_bit_for_bit(cuda_device, kv_len):
    q, k, v = make_qkv(1, kv_len, seed=kv_len + 3)
    _, _, _, _, _, v8, vs, vstride = quantize_all_gpu(q, k, v)
    vc, vsc = oracle.quantize_v_e4m3(v)
    assert np.array_equal(vs.cpu().numpy(), vsc)
    assert np.array_equal(v8[:, :, :kv_len].cpu().numpy(), vc.transpose(1, 2, 0))
    assert torch.all(v8[:, :, kv_len:] == 0x7F)  # past kv_len: untouched


@pytest.mark.parametrize("q_len,kv_len", [(1, 1), (5, 300), (43, 300), (100, 100), (129, 1000),
                                          (22, 2000)])
@pytest.mark.parametrize("variant", [1, 2])
def test_fp8pv_small_shapes_every_element(cuda_device, q_len, kv_len, variant):
    q, k, v = make_qkv(q_len, kv_len, seed=29 * q_len + kv_len)
    out, lse, plan = run_fp8pv(q, k, v, SCALE, force_variant=variant)
    assert plan["variant"] == variant
    ref_o, ref_l, bound = oracle_fp8pv(q, k, v, SCALE)
    got = out.double().cpu().numpy()
    check_pv(got, lse.double().cpu().numpy(), ref_o, ref_l, bound, f"fp8pv {q_len}x{kv_len}")
    if q_len == kv_len:
        # token 0 sees key 0 alone: its probability is exactly 1 (stored 2^6, exact in
        # E4M3), so it returns the dequantised V row up to BF16 rounding
        vc, vs = oracle.quantize_v_e4m3(v)
        want = np.repeat(oracle.dequantize_v_e4m3(vc, vs)[0], 6, axis=0)
        assert np.all(np.abs(got[0] - want) <= 2.0 ** -8 * np.abs(want) + 1e-7)


@pytest.mark.parametrize("splits,grid,variant", [(3, 0, 1), (3, 5, 1), (2, 0, 2), (3, 6, 2),
                                                 (32, 0, 1), (-1, 0, 1), (-1, 6, 2)])
def test_fp8pv_split_tail_every_element(cuda_device, splits, grid, variant):
    q, k, v = make_qkv(129, 1000, seed=37)
    out, lse, _ = run_fp8pv(q, k, v, SCALE, force_splits=splits, force_grid=grid,
                            force_variant=variant)
    ref_o, ref_l, bound = oracle_fp8pv(q, k, v, SCALE)
    check_pv(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l, bound,
             f"fp8pv split {splits} grid {grid}")


@pytest.mark.parametrize("variant", [1, 2])
def test_fp8pv_equal_scores_give_the_mean_of_dequantised_v(cuda_device, variant):
    """Q = 0: every visible key gets the same probability, exactly representable in
    E4M3, so the output is the mean of the visible dequantised V rows (channel
    scale applied per column) up to FP32 sums and BF16 rounding."""
    q, k, v = make_qkv(50, 700, seed=41)
    q = torch.zeros_like(q)
    out, lse, _ = run_fp8pv(q, k, v, SCALE, force_variant=variant)
    vc, vs = oracle.quantize_v_e4m3(v)
    vd = oracle.dequantize_v_e4m3(vc, vs)
    p0 = 700 - 50
    got = out.double().cpu().numpy()
    for t in (0, 1, 20, 49):
        mean = vd[:p0 + t + 1].mean(axis=0)  # [4, 256]
        want = np.repeat(mean, 6, axis=0)    # query head h reads KV head h // 6
        assert np.all(np.abs(got[t] - want) <= 2.0 ** -8 * np.abs(want) + 1e-5), t
        assert np.allclose(lse[t].cpu().numpy(), np.log(p0 + t + 1), atol=1e-5)


@pytest.mark.parametrize("name", ["q4096_kv32768", "q512_kv4096_kbias", "q3072_kv16384"])
@pytest.mark.parametrize("variant", [0, 1])
def test_fp8pv_workload_full_size(cuda_device, name, variant):
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    out, lse, plan = run_fp8pv(q, k, v, w.scale, force_variant=variant)
    rows = item_cover_rows(w.q_len, w.n_q_heads, sample_rows(w.q_len, w.n_q_heads, 600, seed=13))
    assert unchecked_items(rows, w.q_len, 21 * plan["variant"]) == []
    ref_o, ref_l, bound = oracle_fp8pv(q, k, v, w.scale, rows=rows)
    got_o, got_l = gather_rows(out, lse, rows)
    err = check_pv(got_o, got_l, ref_o, ref_l, bound, f"fp8pv {name}")
    # long rows: the P rounding errors are many and of both signs; on average they
    # stay within the BF16 path's acceptance mean
    assert err.mean() <= 2e-3


def test_fp8pv_refusals(cuda_device):
    import gqa_chunked_prefill_gb300 as gqa
    S = gqa.GqaStatus
    q8, qs, k8, ks, kstride, v8, vs, vstride = quantize_all_gpu(*make_qkv(8, 40, seed=1))
    out = torch.empty((8, 24, 256), dtype=torch.bfloat16, device="cuda")
    f = lambda **kw: gqa.gqa_prefill_attn_fp8qkpv(
        q8, qs, k8, ks, kstride, v8, kw.get("vs", vs), kw.get("vstride", vstride), out, None, 8,
        kw.get("kv", 40), 24, 4, 256, SCALE, check=False)
    assert f(vstride=24) == S.ERR_SHAPE      # not a multiple of 16
    assert f(vstride=32) == S.ERR_SHAPE      # shorter than kv_len
    assert f(vs=None) == S.ERR_NULL
    assert gqa.gqa_quantize_v_fp8(v8, v8, vs, 40, 4, 256, 40, check=False) == S.ERR_SHAPE
    assert f() == S.OK
    torch.cuda.synchronize()


def test_fp8pv_method_error_against_bf16_attention(cuda_device):
    """Not parity: the method's own error on N(0, 1) data, against unquantised
    attention. E4M3 Q, K, V and P each carry about 2^-4 relative rounding."""
    q, k, v = make_qkv(64, 2000, seed=78)
    out, lse, _ = run_fp8pv(q, k, v, SCALE)
    ref_o, ref_l = oracle.attention(q, k, v, SCALE)
    err = np.abs(out.double().cpu().numpy() - ref_o)
    assert err.mean() < 1e-2 and err.max() < 2e-1
    assert np.abs(lse.double().cpu().numpy() - ref_l).max() < 5e-2
