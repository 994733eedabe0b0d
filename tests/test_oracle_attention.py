"""Pins for oracle.attention: a library routine (torch SDPA in float64), closed-form
special cases, block-table permutation and block-size invariance."""

import os

import numpy as np
import pytest
import torch

from oracle import attention, cache, numerics

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _build(ctx_lens, hkv, d, bs, tables, nb, dtype, rng, poison=False):
    """Pools filled through append + slot mapping, and the logical K/V per sequence."""
    kp = cache.new_pool(nb, hkv, bs, d, dtype)
    vp = cache.new_pool(nb, hkv, bs, d, dtype)
    if poison:
        kp.view(np.uint8)[...] = 0xFF          # NaN in every float type
        vp.view(np.uint8)[...] = 0xFF
    Ks, Vs = [], []
    for s, c in enumerate(ctx_lens):
        k = numerics.store(rng.normal(size=(c, hkv, d)).astype(np.float32), "f32", dtype)
        v = numerics.store(rng.normal(size=(c, hkv, d)).astype(np.float32), "f32", dtype)
        slots = cache.slot_mapping(tables, [s] * c, range(c), bs)
        cache.kv_append(kp, vp, k, v, slots, dtype, dtype)
        Ks.append(numerics.to_f64(k, dtype))
        Vs.append(numerics.to_f64(v, dtype))
    return kp, vp, Ks, Vs


def _sdpa(q, K, V, scale):
    """torch scaled_dot_product_attention on CPU float64, KV heads repeated per group."""
    hq, d = q.shape
    ctx, hkv, _ = K.shape
    g = hq // hkv
    Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(g, dim=0)   # [Hq, ctx, D]
    Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(g, dim=0)
    qt = torch.from_numpy(q)[:, None, :]                                      # [Hq, 1, D]
    out = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    return out[:, 0, :].numpy()


def test_tiny_matches_torch_sdpa_and_paged_equals_contiguous():
    rng = np.random.default_rng(0)
    ctx = [5, 17, 33, 64]
    hq, hkv, d, bs, nb = 4, 2, 64, 16, 32
    perm = rng.permutation(nb)
    tables = np.zeros((4, 4), dtype=np.int32)
    pos = 0
    for s, c in enumerate(ctx):
        n = -(-c // bs)
        tables[s, :n] = perm[pos:pos + n]
        pos += n
    kp, vp, Ks, Vs = _build(ctx, hkv, d, bs, tables, nb, "f32", rng)
    q = rng.normal(size=(4, hq, d)).astype(np.float32)
    out = attention.decode_attention_paged(q, kp, vp, tables, ctx, 0.125, "f32")
    for s in range(4):
        contiguous = attention.decode_attention_contiguous(q[s], Ks[s], Vs[s], 0.125)
        assert np.array_equal(out[s], contiguous)
        np.testing.assert_allclose(out[s], _sdpa(q[s].astype(np.float64), Ks[s], Vs[s], 0.125),
                                   rtol=0, atol=1e-13)


def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(1)
    q = rng.normal(size=(8, 16))
    K = rng.normal(size=(1, 2, 16))
    V = rng.normal(size=(1, 2, 16))
    out = attention.decode_attention_contiguous(q, K, V, 0.3)
    for h in range(8):
        assert np.array_equal(out[h], V[0, h // 4])


def test_equal_keys_average_the_values():
    rng = np.random.default_rng(2)
    q = rng.normal(size=(2, 8))
    K = np.repeat(rng.normal(size=(1, 1, 8)), 50, axis=0)
    V = rng.normal(size=(50, 1, 8))
    out = attention.decode_attention_contiguous(q, K, V, 1.0)
    np.testing.assert_allclose(out, np.repeat(V.mean(axis=0), 2, axis=0), rtol=0, atol=1e-15)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(3)
    q = np.ones((1, 4))
    K = rng.normal(size=(20, 1, 4)) * 0.01
    K[13, 0, :] = 100.0                       # score 400 vs ~0: weight 1 - O(e^-399)
    V = rng.normal(size=(20, 1, 4))
    out = attention.decode_attention_contiguous(q, K, V, 1.0)
    np.testing.assert_allclose(out[0], V[13, 0], rtol=0, atol=1e-15)


def test_two_tokens_hand_computed():
    q = np.array([[1.0, 2.0]])
    K = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])     # scores 1*s, 2*s
    V = np.array([[[3.0, -1.0]], [[5.0, 7.0]]])
    s = 0.5
    w1, w2 = np.exp(0.5), np.exp(1.0)
    expect = (w1 * V[0, 0] + w2 * V[1, 0]) / (w1 + w2)
    np.testing.assert_allclose(attention.decode_attention_contiguous(q, K, V, s)[0], expect,
                               rtol=1e-15, atol=0)


def test_grouping_maps_consecutive_query_heads_to_a_kv_head():
    # reading: with G = Hq/Hkv, query head h reads KV head h // G
    rng = np.random.default_rng(4)
    q = rng.normal(size=(6, 8))
    K = rng.normal(size=(9, 3, 8))
    V = rng.normal(size=(9, 3, 8))
    out = attention.decode_attention_contiguous(q, K, V, 0.2)
    for h in range(6):
        single = attention.decode_attention_contiguous(q[h:h + 1], K[:, h // 2:h // 2 + 1], V[:, h // 2:h // 2 + 1], 0.2)
        assert np.array_equal(out[h], single[0])


def test_block_table_permutation_invariance_with_the_diagram():
    rows = []
    with open(os.path.join(GOLDEN, "block_table_diagram.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    diagram = [int(r[3]) for r in rows]                     # 84, 12, 903
    rng = np.random.default_rng(5)
    hkv, d, bs, ctx = 2, 16, 16, 48
    k = rng.normal(size=(ctx, hkv, d)).astype(np.float32)
    v = rng.normal(size=(ctx, hkv, d)).astype(np.float32)
    q = rng.normal(size=(1, 4, d)).astype(np.float32)
    outs = []
    for table in ([0, 1, 2], diagram, [903, 84, 12]):
        kp = cache.new_pool(904, hkv, bs, d, "f32")
        vp = cache.new_pool(904, hkv, bs, d, "f32")
        slots = cache.slot_mapping([table], [0] * ctx, range(ctx), bs)
        cache.kv_append(kp, vp, k, v, slots, "f32", "f32")
        outs.append(attention.decode_attention_paged(q, kp, vp, [table], [ctx], 0.25, "f32"))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


@pytest.mark.parametrize("ctx", [1, 15, 16, 17, 70])
def test_block_size_invariance(ctx):
    rng = np.random.default_rng(ctx)
    hkv, d = 2, 8
    k = rng.normal(size=(ctx, hkv, d)).astype(np.float32)
    v = rng.normal(size=(ctx, hkv, d)).astype(np.float32)
    q = rng.normal(size=(1, 4, d)).astype(np.float32)
    outs = []
    for bs in (8, 16, 32):
        n = -(-ctx // bs)
        nb = n + 5
        table = list(rng.permutation(nb)[:n])
        kp = cache.new_pool(nb, hkv, bs, d, "f32")
        vp = cache.new_pool(nb, hkv, bs, d, "f32")
        cache.kv_append(kp, vp, k, v, cache.slot_mapping([table], [0] * ctx, range(ctx), bs), "f32", "f32")
        outs.append(attention.decode_attention_paged(q, kp, vp, [table], [ctx], 0.3, "f32"))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_poisoned_unused_slots_are_never_read():
    rng = np.random.default_rng(6)
    ctx = [3, 16, 29]
    tables = np.array([[4, 0], [1, 0], [2, 5]], dtype=np.int32)
    kp, vp, Ks, Vs = _build(ctx, 1, 8, 16, tables, 6, "bf16", rng, poison=True)
    q = numerics.store(rng.normal(size=(3, 2, 8)).astype(np.float32), "f32", "bf16")
    out = attention.decode_attention_paged(q, kp, vp, tables, ctx, 0.35, "bf16", q_dtype="bf16")
    assert np.all(np.isfinite(out))


def test_empty_sequence_outputs_zero():
    out = attention.decode_attention_contiguous(np.ones((2, 4)), np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), 1.0)
    assert np.array_equal(out, np.zeros((2, 4)))


def test_fp8_uses_dequantised_values():
    rng = np.random.default_rng(7)
    codes_k = rng.integers(0, 0x7E, size=(1, 1, 16, 8), dtype=np.uint8)
    codes_v = rng.integers(0, 0x7E, size=(1, 1, 16, 8), dtype=np.uint8)
    q = rng.normal(size=(1, 2, 8)).astype(np.float32)
    sk, sv = np.float32(0.02), np.float32(0.5)
    out = attention.decode_attention_paged(q, codes_k, codes_v, [[0]], [11], 0.3, "fp8_e4m3", sk, sv)
    K = torch.from_numpy(codes_k[0, 0, :11].copy()).view(torch.float8_e4m3fn).double().numpy() * float(sk)
    V = torch.from_numpy(codes_v[0, 0, :11].copy()).view(torch.float8_e4m3fn).double().numpy() * float(sv)
    np.testing.assert_allclose(out[0], _sdpa(q[0].astype(np.float64), K[:, None, :], V[:, None, :], 0.3),
                               rtol=0, atol=1e-12)
