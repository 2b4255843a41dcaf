"""Pins for the FP64 oracle: each test checks it against something other than
itself — a closed form, a textbook library routine, an invariant the method
must satisfy, or an independent numpy restatement — so that a dropped term, a
wrong sign, a wrong index or a transposed operand in the oracle fails here.

Definition pinned: QK^T, bottom-right causal mask, softmax and PV
(DCU使用技术报告（中篇）, §2), query head h on KV head h/6
(gfx936 DCU上实现INT8 QK MMAC, §5.2), LSE = natural log of the softmax
normaliser of the scaled scores.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import restate_numpy as rn
from gqa_inputs import make_qkv

SCALE = 1.0 / 16.0


def rand64(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --- closed forms ---------------------------------------------------------------

def test_single_key_returns_v_and_dot_lse():
    q, k, v = rand64((1, 24, 256), 1), rand64((1, 4, 256), 2), rand64((1, 4, 256), 3)
    out, lse = oracle.attention(q, k, v, SCALE)
    for h in range(24):
        g = h // 6
        assert np.array_equal(out[0, h], v[0, g])  # e = 1, Z = 1: exact
        assert abs(lse[0, h] - SCALE * float(np.dot(q[0, h], k[0, g]))) < 1e-12


def test_first_row_of_unprefixed_chunk_returns_v0():
    q, k, v = rand64((7, 24, 256), 4), rand64((7, 4, 256), 5), rand64((7, 4, 256), 6)
    out, _ = oracle.attention(q, k, v, SCALE)
    for h in range(24):
        assert np.array_equal(out[0, h], v[0, h // 6])


@pytest.mark.parametrize("zero", ["q", "k"])
def test_constant_scores_give_mean_of_visible_v(zero):
    q_len, kv_len = 5, 11
    q, k, v = rand64((q_len, 24, 64), 7), rand64((kv_len, 4, 64), 8), rand64((kv_len, 4, 64), 9)
    if zero == "q":
        q[:] = 0.0
    else:
        k[:] = 0.0
    out, lse = oracle.attention(q, k, v, SCALE)
    for t in range(q_len):
        p = kv_len - q_len + t
        for h in range(24):
            np.testing.assert_allclose(out[t, h], v[: p + 1, h // 6].mean(axis=0), rtol=0, atol=1e-13)
            assert abs(lse[t, h] - math.log(p + 1)) < 1e-13


def test_linear_scores_geometric_series():
    """q = a*e0, k_j = j*e0, v_j = j: scores c*j with c = scale*a; the output is the
    mean key index under weights e^{c j}, j = 0..p, and lse = ln sum_j e^{c j}."""
    q_len, kv_len, d, a = 6, 40, 32, 3.0
    q = np.zeros((q_len, 24, d)); q[:, :, 0] = a
    k = np.zeros((kv_len, 4, d)); k[:, :, 0] = np.arange(kv_len)[:, None]
    v = np.zeros((kv_len, 4, d)); v[:, :, :] = np.arange(kv_len)[:, None, None]
    scale = 0.05
    c = scale * a
    out, lse = oracle.attention(q, k, v, scale)
    for t in range(q_len):
        p = kv_len - q_len + t
        r = math.exp(c)
        z = (r ** (p + 1) - 1.0) / (r - 1.0)
        # sum_j j r^j for j = 0..p
        num = r * (1 - (p + 1) * r ** p + p * r ** (p + 1)) / (1 - r) ** 2
        for h in range(24):
            assert abs(lse[t, h] - math.log(z)) < 1e-11
            np.testing.assert_allclose(out[t, h], num / z, rtol=1e-12, atol=0)


def test_probabilities_sum_to_one():
    q, k, v = make_qkv(9, 300, 11)
    _, _, psum = oracle.attention(q, k, v, SCALE, with_prob_sum=True)
    assert np.max(np.abs(psum - 1.0)) < 1e-12


# --- invariants -----------------------------------------------------------------

def test_future_keys_do_not_change_earlier_rows():
    q_len, kv_len = 12, 40
    q, k, v = rand64((q_len, 24, 32), 12), rand64((kv_len, 4, 32), 13), rand64((kv_len, 4, 32), 14)
    out, lse = oracle.attention(q, k, v, SCALE)
    t_star = 5
    p_star = kv_len - q_len + t_star
    k2, v2 = k.copy(), v.copy()
    k2[p_star + 1:] += 10.0 * rand64(k2[p_star + 1:].shape, 15)
    v2[p_star + 1:] -= 7.0
    out2, lse2 = oracle.attention(q, k2, v2, SCALE)
    assert np.array_equal(out[: t_star + 1], out2[: t_star + 1])
    assert np.array_equal(lse[: t_star + 1], lse2[: t_star + 1])
    assert not np.array_equal(out[t_star + 1:], out2[t_star + 1:])


def test_per_head_key_shift_moves_lse_only():
    q_len, kv_len = 6, 30
    q, k, v = rand64((q_len, 24, 64), 16), rand64((kv_len, 4, 64), 17), rand64((kv_len, 4, 64), 18)
    b = 0.5 * rand64((4, 64), 19)
    out, lse = oracle.attention(q, k, v, SCALE)
    out2, lse2 = oracle.attention(q, k + b[None], v, SCALE)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-12)
    for h in range(24):
        shift = SCALE * (q[:, h, :] @ b[h // 6])
        np.testing.assert_allclose(lse2[:, h] - lse[:, h], shift, rtol=0, atol=1e-12)


def test_thread_count_and_row_subset_are_bit_identical():
    q, k, v = make_qkv(33, 200, 20)
    out1, lse1 = oracle.attention(q, k, v, SCALE, n_threads=1)
    out8, lse8 = oracle.attention(q, k, v, SCALE, n_threads=8)
    assert np.array_equal(out1, out8) and np.array_equal(lse1, lse8)
    rows = np.array([0, 5, 24 * 7 + 3, 24 * 33 - 1], dtype=np.int64)
    o_r, l_r = oracle.attention(q, k, v, SCALE, rows=rows)
    flat_o, flat_l = out1.reshape(-1, 256), lse1.reshape(-1)
    assert np.array_equal(o_r, flat_o[rows]) and np.array_equal(l_r, flat_l[rows])


# --- independent restatements ---------------------------------------------------

@pytest.mark.parametrize("q_len,kv_len", [(1, 1), (1, 8), (3, 3), (3, 8), (8, 8), (5, 7)])
@pytest.mark.parametrize("hq,hkv,d", [(24, 4, 256), (6, 1, 16), (8, 2, 8)])
def test_brute_force_matches_numpy_replicated_heads(q_len, kv_len, hq, hkv, d):
    seed = 100 * q_len + kv_len + hq
    q, k, v = rand64((q_len, hq, d), seed), rand64((kv_len, hkv, d), seed + 1), rand64((kv_len, hkv, d), seed + 2)
    out, lse = oracle.attention(q, k, v, 0.3)
    out_r, lse_r = rn.gqa_by_replication(q, k, v, 0.3)
    np.testing.assert_allclose(out, out_r, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_r, rtol=1e-12, atol=1e-12)


def _sdpa(q, k, v, scale, mask=None, is_causal=False):
    rep = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)                       # [H, T, d]
    kt = torch.from_numpy(k).repeat_interleave(rep, dim=1).permute(1, 0, 2)
    vt = torch.from_numpy(v).repeat_interleave(rep, dim=1).permute(1, 0, 2)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=mask, is_causal=is_causal, scale=scale)
    return o.permute(1, 0, 2).numpy()


def test_square_chunk_is_textbook_causal_attention():
    """q_len == kv_len: standard causal attention, where torch's top-left
    is_causal alignment coincides with the chunk-at-the-end alignment."""
    q, k, v = rand64((37, 24, 256), 30), rand64((37, 4, 256), 31), rand64((37, 4, 256), 32)
    out, _ = oracle.attention(q, k, v, SCALE)
    np.testing.assert_allclose(out, _sdpa(q, k, v, SCALE, is_causal=True), rtol=1e-10, atol=1e-12)


def test_prefixed_chunk_matches_library_with_bottom_right_mask():
    q_len, kv_len = 13, 50
    q, k, v = rand64((q_len, 24, 64), 33), rand64((kv_len, 4, 64), 34), rand64((kv_len, 4, 64), 35)
    mask = torch.ones(q_len, kv_len, dtype=torch.bool).tril(diagonal=kv_len - q_len)
    out, lse = oracle.attention(q, k, v, SCALE)
    np.testing.assert_allclose(out, _sdpa(q, k, v, SCALE, mask=mask), rtol=1e-10, atol=1e-12)
    # LSE against torch.logsumexp of the masked scaled scores
    qt = torch.from_numpy(q)
    kt = torch.from_numpy(k).repeat_interleave(6, dim=1)
    s = SCALE * torch.einsum("thd,jhd->htj", qt, kt)
    s = s.masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).T.numpy(), rtol=0, atol=1e-12)


def test_bf16_inputs_are_widened_exactly():
    q, k, v = make_qkv(4, 9, 40)
    out_a, lse_a = oracle.attention(q, k, v, SCALE)
    out_b, lse_b = oracle.attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), SCALE)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


def test_rejects_bad_arguments():
    q, k, v = rand64((4, 24, 8), 1), rand64((3, 4, 8), 2), rand64((3, 4, 8), 3)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, SCALE)  # kv_len < q_len


def test_stored_oracle_values_unchanged():
    import os
    from gqa_inputs import WORKLOADS, make_workload
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_q128_kv256.txt")
    lines = [l.split() for l in open(path) if not l.startswith("#")]
    rows = [int(l[0]) for l in lines]
    cols = [0, 1, 128, 255]
    w = WORKLOADS["q128_kv256"]
    q, k, v = make_workload(w)
    out, lse = oracle.attention(q, k, v, w.scale, rows=rows)
    for i, l in enumerate(lines):
        assert abs(lse[i] - float(l[1])) < 1e-12
        for j, c in enumerate(cols):
            assert abs(out[i, c] - float(l[2 + j])) < 1e-12


# --- paged K/V: the block-table gather --------------------------------------------

def test_paged_gather_worked_example_by_hand():
    """page_size 2, three pages whose slots hold 10*page + slot, block table [2, 0, 1]:
    keys 0..4 live at (page 2, slot 0), (2, 1), (0, 0), (0, 1), (1, 0)."""
    cache = np.zeros((3, 2, 1, 1))
    for page in range(3):
        for slot in range(2):
            cache[page, slot, 0, 0] = 10 * page + slot
    k, v = oracle.paged_gather(cache, -cache, [2, 0, 1], kv_len=5)
    assert k[:, 0, 0].tolist() == [20, 21, 0, 1, 10]
    assert v[:, 0, 0].tolist() == [-20, -21, 0, -1, -10]


def test_paged_gather_repeated_page():
    cache = np.arange(8, dtype=np.float64).reshape(2, 4, 1, 1)
    k, _ = oracle.paged_gather(cache, cache, [1, 1], kv_len=7)
    assert k[:, 0, 0].tolist() == [4, 5, 6, 7, 4, 5, 6]


@pytest.mark.parametrize("kv_len,page_size", [(1, 16), (40, 16), (300, 48), (300, 784), (1000, 64)])
def test_paged_gather_inverts_the_cache_scatter(kv_len, page_size):
    """The input generator scatters logical pages to seeded physical pages and
    fills every other slot with NaN; reading the sequence back through the
    table must give the dense K/V bit for bit, and no NaN."""
    from gqa_inputs import make_paged_cache
    q, k, v = make_qkv(min(kv_len, 7), kv_len, 50 + kv_len)
    kc, vc, table = make_paged_cache(k, v, page_size, seed=kv_len + page_size)
    assert kc.shape[0] == -(-kv_len // page_size) + 3
    assert torch.isnan(kc.float()).any()  # unused slots really are poisoned
    k2, v2 = oracle.paged_gather(kc, vc, table, kv_len)
    assert torch.equal(k2, k) and torch.equal(v2, v)
    out_p, lse_p = oracle.paged_attention(q, kc, vc, table, kv_len, SCALE)
    out_d, lse_d = oracle.attention(q, k, v, SCALE)
    assert np.array_equal(out_p, out_d) and np.array_equal(lse_p, lse_d)


def test_paged_gather_rejects_entries_outside_the_cache():
    cache = np.zeros((2, 4, 1, 1))
    with pytest.raises(ValueError):
        oracle.paged_gather(cache, cache, [0, 2], kv_len=6)
    with pytest.raises(ValueError):
        oracle.paged_gather(cache, cache, [-1], kv_len=3)


# --- quantised QK^T: E4M3 codes and per-vector scales -----------------------------

def test_e4m3_values_follow_the_format():
    v = oracle.e4m3_values()
    assert v[0] == 0.0 and v[1] == 2.0 ** -9 and v[7] == 7 * 2.0 ** -9  # subnormals m/8 * 2^-6
    assert v[8] == 2.0 ** -6 and v[0x38] == 1.0 and v[0x3F] == 1.875
    assert v[0x7E] == 448.0 and v[0x7D] == 416.0
    assert np.all(np.diff(v) > 0)


def test_e4m3_every_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes).astype(np.float32)), codes)


def test_e4m3_rounding_by_hand():
    x = [448.0, 1.0, 2.0 ** -9, 2.0 ** -10, 1.0625, 1.1875, 1.125 + 2.0 ** -10, 470.0, 1e30,
         -1.0, -1e-9, 3 * 2.0 ** -10]
    # 2^-10 ties 0 / 2^-9 -> 0 (even); 1.0625 ties 1.0 / 1.125 -> 1.0 (code 0x38, even);
    # 1.1875 ties 1.125 / 1.25 -> 1.25 (0x3A); just above 1.125 -> 0x39; beyond 448 -> 448;
    # -1e-9 rounds to -0 (sign kept); 3*2^-10 ties 2^-9 / 2^-8 -> 2^-8 (code 0x02).
    want = [0x7E, 0x38, 0x01, 0x00, 0x38, 0x3A, 0x39, 0x7E, 0x7E, 0xB8, 0x80, 0x02]
    assert oracle.e4m3_encode(x).tolist() == want


def test_e4m3_matches_library_cast():
    x = (torch.randn(200000, generator=torch.Generator().manual_seed(3)) * 60).clamp(-447, 447)
    lib = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x.numpy()), lib)


def test_quantize_per_vector_scale_and_error_bound():
    q, _, _ = make_qkv(9, 9, 44)
    x = q.float().numpy()
    x[3, 5] = 0.0  # one all-zero vector
    codes, s = oracle.quantize_e4m3(x)
    amax = np.abs(x).max(axis=-1)
    assert s.dtype == np.float32 and np.array_equal(s, (amax / np.float32(448)).astype(np.float32))
    assert np.all(codes[3, 5] == 0) and s[3, 5] == 0
    dq = oracle.dequantize_e4m3(codes, s)
    err = np.abs(dq - x)
    # half a code spacing: 2^-4 relative in the normal range, 2^-10 * s among subnormals
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s[..., None].astype(np.float64)) * 1.0001
    assert np.all(err <= bound)
    # the largest element of every non-zero vector maps to +-448
    nz = amax > 0
    top = np.take_along_axis(oracle.e4m3_decode(codes), np.abs(x).argmax(-1)[..., None], -1)[..., 0]
    assert np.all(np.abs(top[nz]) == 448.0)


def test_fp8qk_attention_equals_attention_on_exact_codes():
    """Integers with max |x| = 448 in every vector quantise exactly (s = 1): the
    quantised path must then equal plain attention on those values."""
    g = np.random.default_rng(9)
    q = g.integers(-16, 17, (5, 24, 256)).astype(np.float64); q[..., 0] = 448
    k = g.integers(-16, 17, (40, 4, 256)).astype(np.float64); k[..., 7] = -448
    v = g.standard_normal((40, 4, 256))
    qc, qs = oracle.quantize_e4m3(q)
    kc, ks = oracle.quantize_e4m3(k)
    assert np.all(qs == 1.0) and np.all(ks == 1.0)
    out_a, lse_a = oracle.fp8qk_attention(qc, qs, kc, ks, v, 1e-5)
    out_b, lse_b = oracle.attention(q, k, v, 1e-5)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


# --- batches of sequences ---------------------------------------------------------

def test_varlen_single_sequence_is_attention():
    q, k, v = make_qkv(9, 40, 61)
    o1, l1 = oracle.varlen_attention(q, k, v, [0, 9], [0, 40], SCALE)
    o2, l2 = oracle.attention(q, k, v, SCALE)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_varlen_sequences_do_not_see_each_other():
    from gqa_inputs import make_varlen
    q, k, v, cu_q, cu_k = make_varlen([(5, 30), (0, 7), (8, 8), (3, 50)], 70)
    out, lse = oracle.varlen_attention(q, k, v, cu_q, cu_k, SCALE)
    k2, v2 = k.clone(), v.clone()
    k2[cu_k[2]:cu_k[3]] = 3.0  # change only sequence 2's keys and values
    v2[cu_k[2]:cu_k[3]] = -1.0
    out2, lse2 = oracle.varlen_attention(q, k2, v2, cu_q, cu_k, SCALE)
    rows2 = slice(cu_q[2], cu_q[3])
    keep = np.ones(out.shape[0], bool)
    keep[rows2] = False
    assert np.array_equal(out[keep], out2[keep]) and np.array_equal(lse[keep], lse2[keep])
    assert not np.array_equal(out[rows2], out2[rows2])


def test_varlen_matches_library_per_sequence_bottom_right_masks():
    from gqa_inputs import make_varlen
    q, k, v, cu_q, cu_k = make_varlen([(4, 20), (6, 6), (1, 33)], 80)
    out, _ = oracle.varlen_attention(q, k, v, cu_q, cu_k, SCALE)
    for b in range(3):
        qb = q[cu_q[b]:cu_q[b + 1]].double().numpy()
        kb = k[cu_k[b]:cu_k[b + 1]].double().numpy()
        vb = v[cu_k[b]:cu_k[b + 1]].double().numpy()
        ql, kl = qb.shape[0], kb.shape[0]
        mask = torch.ones(ql, kl, dtype=torch.bool).tril(diagonal=kl - ql)
        np.testing.assert_allclose(out[cu_q[b]:cu_q[b + 1]], _sdpa(qb, kb, vb, SCALE, mask=mask),
                                   rtol=1e-10, atol=1e-12)


def test_paged_batch_scatter_is_read_back_exactly():
    from gqa_inputs import make_paged_batch, make_varlen
    q, k, v, cu_q, cu_k = make_varlen([(3, 100), (0, 17), (5, 5), (2, 260)], 90)
    kc, vc, table, kv_lens = make_paged_batch(k, v, cu_k, 48, seed=91)
    for b, kl in enumerate(kv_lens):
        kb, vb = oracle.paged_gather(kc, vc, table[b], kl)
        assert torch.equal(kb, k[cu_k[b]:cu_k[b + 1]]) and torch.equal(vb, v[cu_k[b]:cu_k[b + 1]])
    o1, l1 = oracle.paged_varlen_attention(q, kc, vc, table, cu_q, kv_lens, SCALE)
    o2, l2 = oracle.varlen_attention(q, k, v, cu_q, cu_k, SCALE)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# --- quantised PV ---------------------------------------------------------------

def test_v_channel_scales_and_codes_by_hand():
    """Channel c of KV head g over all keys is one vector: its scale is its largest
    magnitude / 448 and each value's code is E4M3(v / s). Worked by hand on a
    3-key, 1-head, 2-channel V (channel 1 is all zeros: scale 0, codes 0)."""
    v = np.zeros((3, 1, 2), np.float32)
    v[:, 0, 0] = [1.0, -2.0, 0.5]          # max |v| = 2: s = 2 / 448 = 1 / 224
    codes, s = oracle.quantize_v_e4m3(v)
    assert s.shape == (1, 2) and s[0, 0] == np.float32(2.0) / np.float32(448.0) and s[0, 1] == 0
    # 1 / s = 224 (E4M3 224 = 1.75 * 2^7: e=14, m=6 -> 0x76); -2 / s = -448 (0xFE);
    # 0.5 / s = 112 (1.75 * 2^6: 0x6E)
    assert list(codes[:, 0, 0]) == [0x76, 0xFE, 0x6E]
    assert list(codes[:, 0, 1]) == [0, 0, 0]
    np.testing.assert_array_equal(oracle.dequantize_v_e4m3(codes, s)[:, 0, 0],
                                  np.array([224.0, -448.0, 112.0]) * float(s[0, 0]))


def test_v_quantisation_is_the_vector_rule_along_keys():
    """The V rule is quantize_e4m3 applied to each (head, channel) column over keys,
    not to each key's 256 values: transposing first gives the same codes."""
    v = rand64((37, 4, 256), 71).astype(np.float32)
    codes, s = oracle.quantize_v_e4m3(v)
    for g in range(4):
        for c in (0, 17, 255):
            cc, ss = oracle.quantize_e4m3(v[:, g, c][None, :])
            np.testing.assert_array_equal(codes[:, g, c], cc[0])
            assert s[g, c] == ss[0] == np.float32(np.abs(v[:, g, c]).max()) / np.float32(448.0)
    per_key, _ = oracle.quantize_e4m3(v)  # the Q/K rule would differ
    assert not np.array_equal(per_key, codes)


def test_fp8pv_attention_equals_attention_on_exact_codes():
    """Values that are already codes times a power-of-two channel scale (each
    channel reaching +-448 times its scale) survive quantisation exactly, so the
    quantised-PV result is plain attention on them."""
    rng = np.random.default_rng(5)
    q_len, kv_len = 6, 40
    q = rand64((q_len, 24, 256), 1)
    k = rand64((kv_len, 4, 256), 2)
    vals = oracle.e4m3_values()
    cv = rng.choice(vals, size=(kv_len, 4, 256)) * rng.choice([-1.0, 1.0], size=(kv_len, 4, 256))
    cv[0] = 448.0  # every channel reaches the largest code
    v = cv * (2.0 ** rng.integers(-8, 3, size=(1, 4, 256)))
    vc, vs = oracle.quantize_v_e4m3(v)
    np.testing.assert_array_equal(oracle.dequantize_v_e4m3(vc, vs), v)
    qc, qs = oracle.quantize_e4m3(q)
    kc, ks = oracle.quantize_e4m3(k)
    got_o, got_l = oracle.fp8pv_attention(qc, qs, kc, ks, vc, vs, SCALE)
    ref_o, ref_l = oracle.attention(oracle.dequantize_e4m3(qc, qs), oracle.dequantize_e4m3(kc, ks),
                                    v, SCALE)
    np.testing.assert_array_equal(got_o, ref_o)
    np.testing.assert_array_equal(got_l, ref_l)


def test_power_of_two_channel_scale_scales_the_output_column():
    """Scaling one V channel by 2^k leaves its codes alone, multiplies its scale by
    2^k and the output column by exactly 2^k; the other columns do not move."""
    q, k, v = (t.double().numpy() for t in make_qkv(9, 50, seed=61))
    vc, vs = oracle.quantize_v_e4m3(v)
    v2 = v.copy()
    v2[:, 2, 77] *= 2.0 ** 5
    vc2, vs2 = oracle.quantize_v_e4m3(v2)
    np.testing.assert_array_equal(vc2, vc)
    assert vs2[2, 77] == vs[2, 77] * 32 and np.array_equal(np.delete(vs2.ravel(), 2 * 256 + 77),
                                                           np.delete(vs.ravel(), 2 * 256 + 77))
    qc, qs = oracle.quantize_e4m3(q)
    kc, ks = oracle.quantize_e4m3(k)
    o1, _ = oracle.fp8pv_attention(qc, qs, kc, ks, vc, vs, SCALE)
    o2, _ = oracle.fp8pv_attention(qc, qs, kc, ks, vc2, vs2, SCALE)
    np.testing.assert_array_equal(o2[:, 12:18, 77], o1[:, 12:18, 77] * 32)  # heads of group 2
    mask = np.ones(o1.shape, bool)
    mask[:, 12:18, 77] = False
    np.testing.assert_array_equal(o2[mask], o1[mask])


def _online_p_rounding(q, k, v, scale, t, h, rng, tile=16, threshold=2.0, pscale=6.0):
    """Brute force of the method's PV for one row: keys in tiles, a running maximum
    (log2 units) raised only when it grows by more than `threshold`, P stored as
    E4M3(2^(x - m + pscale)), O and the row sum rescaled when m moves."""
    kv_len = k.shape[0]
    p_last = kv_len - q.shape[0] + t
    g = h // (q.shape[1] // k.shape[1])
    x = scale * (k[:p_last + 1, g] @ q[t, h]) / math.log(2.0)
    m, o, l = -np.inf, np.zeros(v.shape[2]), 0.0
    for a in range(0, p_last + 1, tile):
        xt = x[a:a + tile]
        if xt.max() > m + threshold:
            m_new = xt.max() + rng.uniform(-threshold, 0)  # any reference at most `threshold` low
            m_new = max(m_new, xt.max() - threshold)
            if np.isfinite(m):
                o *= 2.0 ** (m - m_new)
                l *= 2.0 ** (m - m_new)
            m = m_new
        pf = 2.0 ** (xt - m + pscale)
        pq = oracle.e4m3_decode(oracle.e4m3_encode(pf.astype(np.float32)))
        o += pq @ v[a:a + len(xt), g]
        l += pf.sum()
    return o / l


def test_p_rounding_stays_within_the_bound():
    """The E4M3 rounding of P, simulated key by key with running maxima anywhere in
    the allowed band, never moves an output element by more than fp8pv_p_bound;
    and the bound is not slack by orders of magnitude (the worst case uses a good
    part of it)."""
    rng = np.random.default_rng(9)
    q, k, v = (t.double().numpy() for t in make_qkv(5, 300, seed=62))
    k[100:110] *= 4.0  # a few large scores: peaked rows and rescales
    rows = np.array([0, 24 * 2 + 7, 24 * 4 + 23])
    ref_o, _ = oracle.attention(q, k, v, SCALE, rows=rows)
    bound = oracle.fp8pv_p_bound(q, k, v, SCALE, rows=rows)
    worst = 0.0
    for i, r in enumerate(rows):
        for _ in range(3):
            got = _online_p_rounding(q, k, v, SCALE, r // 24, r % 24, rng)
            err = np.abs(got - ref_o[i])
            assert np.all(err <= bound[i] * (1 + 1e-9)), (r, (err / bound[i]).max())
            worst = max(worst, (err / bound[i]).max())
    assert worst > 0.05


def test_p_bound_by_hand():
    """Two visible keys with scores 0 and ln(1/2) (p = 1, 1/2), one channel with
    v = (1, -3): B = ((2^-4 + 2^-16) * 1 + (2^-4 / 2 + 2^-16) * 3) / 1.5."""
    q = np.zeros((1, 1, 1))
    q[0, 0, 0] = 1.0
    k = np.array([[[0.0]], [[math.log(0.5)]]])
    v = np.array([[[1.0]], [[-3.0]]])
    b = oracle.fp8pv_p_bound(q, k, v, 1.0)
    want = ((2 ** -4 + 2 ** -16) * 1 + (2 ** -5 + 2 ** -16) * 3) / 1.5
    assert abs(b[0, 0, 0] - want) < 1e-15


def test_p_bound_needs_its_subnormal_term():
    """One dominant key and 200000 keys whose stored P (2^6 * p) is 0.45 * 2^-9,
    below half the smallest E4M3 subnormal: they all round to zero although they
    carry most of the row's mass. The bound holds; its relative term alone (what
    a normal-range-only analysis would give) does not."""
    kv_len = 200001
    q = np.zeros((1, 1, 8))
    q[0, 0, 0] = 1.0
    k = np.zeros((kv_len, 1, 8))
    k[1:, 0, 0] = (math.log2(0.45) - 9 - 6) * math.log(2.0)  # 2^6 * p = 0.45 * 2^-9
    v = np.ones((kv_len, 1, 8))
    v[:, 0, 1:] = np.linspace(0.5, 2.0, 7)
    ref_o, _ = oracle.attention(q, k, v, 1.0)
    got = _online_p_rounding(q, k, v, 1.0, 0, 0, np.random.default_rng(3), tile=kv_len,
                             threshold=0.0)
    err = np.abs(got - ref_o[0, 0])
    bound = oracle.fp8pv_p_bound(q, k, v, 1.0)[0, 0]
    assert np.all(err <= bound)
    p = np.exp(k[:, 0, 0] - k[:, 0, 0].max())
    rel_only = (oracle.E4M3_P_REL * p @ v[:, 0]) / p.sum()
    assert np.all(err > 5 * rel_only)
