"""Pins the fp64 oracle to things other than itself (CPU only).

Each pin is chosen so that a plausible slip in the oracle fails it:
  * number formats: torch's float->bf16 rounding, hand-picked ties, a double-rounding trap;
  * RoPE: complex multiplication by e^{i*angle} (numpy), norm, relative-position invariance;
  * decode: two 3-token cases worked out in closed form, and special cases that reduce to
    torch's scaled_dot_product_attention (Shared KV = M_h = I with no positional slice,
    plain GQA, the key materialised from the page's K_h = V_g M_h);
  * head->group map, split-T invariance, ragged tails, the paged layout and the
    cache-size closed form against the figures the pages print;
  * the fp8 value cache (a reading of this library's, not the pages'): torch's E4M3 format
    on every code and on every tie, the scale exponent's closed form, the quantised append,
    and decode over fp8 codes equal to decode over the values torch dequantises from them.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from compact_kv_cache_gva_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f(bits):
    return torch.tensor(np.asarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)


# ---------------------------------------------------------------- number formats

def test_bf16_encode_matches_torch_on_f32_values(oracle_mod):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(4000), rng.standard_normal(1000) * 1e-30,
                        rng.standard_normal(1000) * 1e30]).astype(np.float32)
    want = bf16_bits(x)
    got = np.array([oracle_mod.double_to_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_ties_and_double_rounding(oracle_mod):
    # ties go to the even significand
    assert oracle_mod.double_to_bf16(1.0) == 0x3F80
    assert oracle_mod.double_to_bf16(1.0 + 2.0 ** -8) == 0x3F80       # tie, even is down
    assert oracle_mod.double_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82   # tie, even is up
    assert oracle_mod.double_to_bf16(-(1.0 + 3 * 2.0 ** -8)) == 0xBF82
    # just above a tie: must round up; a detour through binary32 would land on the tie
    # (2^-30 is below half a binary32 ulp at 1.0) and round down to even
    assert oracle_mod.double_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert oracle_mod.double_to_bf16(0.0) == 0x0000
    assert oracle_mod.double_to_bf16(-0.0) == 0x8000
    assert oracle_mod.double_to_bf16(1e39) == 0x7F80


def test_bf16_decode_matches_torch(oracle_mod):
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    want = bits_to_f(bits)
    got = np.array([oracle_mod.bf16_to_double(int(b)) for b in bits])
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.isnan(got), np.isnan(want))


# ---------------------------------------------------------------- RoPE

@pytest.mark.parametrize("d_r", [2, 16, 24])
def test_rope_is_complex_rotation(oracle_mod, d_r):
    rng = np.random.default_rng(d_r)
    x = rng.standard_normal(d_r)
    for pos in [0, 1, 7, 4095, 131071]:
        y = oracle_mod.rope(x, pos)
        i = np.arange(d_r // 2)
        ang = pos * 10000.0 ** (-2.0 * i / d_r)
        z = (x[0::2] + 1j * x[1::2]) * np.exp(1j * ang)
        assert np.allclose(y[0::2], z.real, atol=1e-12) and np.allclose(y[1::2], z.imag, atol=1e-12)


def test_rope_norm_and_relative_position(oracle_mod):
    rng = np.random.default_rng(3)
    d_r = 16
    q, k = rng.standard_normal(d_r), rng.standard_normal(d_r)
    for p, j, shift in [(5, 2, 11), (1000, 0, 77), (300, 299, 100000)]:
        base_dot = oracle_mod.rope(q, p) @ oracle_mod.rope(k, j)
        shifted = oracle_mod.rope(q, p + shift) @ oracle_mod.rope(k, j + shift)
        assert abs(base_dot - shifted) < 1e-9
        assert abs(np.linalg.norm(oracle_mod.rope(k, j)) - np.linalg.norm(k)) < 1e-12


# ---------------------------------------------------------------- hand cases

def _one_group_pool(vals, krs, dtype=np.float32):
    """Tiny cache with one block: V rows `vals` [T,d_v], rotated keys `krs` [T,d_r]."""
    T, d_v = vals.shape
    d_r = krs.shape[1] if krs is not None else 0
    vp = np.zeros((1, 1, 64, d_v), dtype=dtype)
    vp[0, 0, :T] = vals
    kp = np.zeros((1, 64, max(d_r, 1)), dtype=dtype)[:, :, :d_r].copy()
    if d_r:
        kp[0, :T] = krs
    return vp, kp


def test_hand_case_A_no_positional_term(oracle_mod):
    # H=G=1, d_v=d_n=2, d_r=2, M=I, scale 1/sqrt(4); v_j=(j,0); q_c=(1,0); q_r=0; query at 2
    vals = np.array([[0, 0], [1, 0], [2, 0]], dtype=np.float64)
    vp, kp = _one_group_pool(vals, np.zeros((3, 2)))
    q_abs, q_rot = oracle_mod.absorb(np.array([[[1.0, 0.0]]]), np.zeros((1, 1, 2)), [2], np.eye(2)[None])
    out = oracle_mod.decode(q_abs, q_rot, vp, kp, np.array([[0]]), [3], G=1, d_n=2)
    s = np.array([0.0, 0.5, 1.0])
    p = np.exp(s) / np.exp(s).sum()
    assert np.allclose(p, [0.186323723226, 0.307195885718, 0.506480391056], atol=1e-12)
    assert abs(out[0, 0, 0] - (p[1] + 2 * p[2])) < 1e-14 and out[0, 0, 1] == 0.0
    assert abs(out[0, 0, 0] - 1.320156667830) < 1e-11


def test_hand_case_B_positional_term(oracle_mod):
    # as A, plus q_r=(1,0) and every raw k_r=(1,0) written at its own position by append;
    # with theta_0 = 1 the positional term of key j is cos(2 - j)
    d_v, d_r = 2, 2
    vals = np.array([[[0, 0]], [[1, 0]], [[2, 0]]], dtype=np.float32)[None]  # [1,3,1,2]
    kr_raw = np.tile(np.array([1.0, 0.0], dtype=np.float32), (1, 3, 1))
    vp = np.zeros((1, 1, 64, d_v), dtype=np.float32)
    kp = np.zeros((1, 64, d_r), dtype=np.float32)
    oracle_mod.append(vals, kr_raw, [0], np.array([[0]]), vp, kp)
    q_abs, q_rot = oracle_mod.absorb(np.array([[[1.0, 0.0]]]), np.array([[[1.0, 0.0]]]), [2], np.eye(2)[None])
    out = oracle_mod.decode(q_abs, q_rot, vp, kp, np.array([[0]]), [3], G=1, d_n=2)
    s = 0.5 * (np.array([0.0, 1.0, 2.0]) + np.cos(2.0 - np.arange(3)))
    assert np.allclose(s, [-0.208073418274, 0.770151152934, 1.5], atol=1e-12)
    p = np.exp(s) / np.exp(s).sum()
    assert np.allclose(p, [0.108955610521, 0.289792493605, 0.601251895873], atol=1e-9)
    # keys were rotated to positions 0,1,2 and rounded to f32 in the cache
    assert abs(out[0, 0, 0] - (p[1] + 2 * p[2])) < 1e-7
    assert abs(out[0, 0, 0] - 1.492296285352) < 1e-7


def test_hand_case_two_queries_causal(oracle_mod):
    # the cache of case B (keys rotated at positions 0,1,2) read by two query tokens, the last
    # two positions: query 0 at position 1 sees keys 0..1 only, with positional terms
    # cos(1 - j):  s = 0.5 * ((0, 1) + (cos 1, 1)) = (0.270151152934, 1.0), so
    # p_1 = e^1 / (e^0.270151 + e^1) = 0.674772102235 and o = (p_1 * 1, 0);
    # query 1 at position 2 is case B itself
    d_v, d_r = 2, 2
    vals = np.array([[[0, 0]], [[1, 0]], [[2, 0]]], dtype=np.float32)[None]
    kr_raw = np.tile(np.array([1.0, 0.0], dtype=np.float32), (1, 3, 1))
    vp = np.zeros((1, 1, 64, d_v), dtype=np.float32)
    kp = np.zeros((1, 64, d_r), dtype=np.float32)
    oracle_mod.append(vals, kr_raw, [0], np.array([[0]]), vp, kp)
    q_abs, q_rot = oracle_mod.absorb(np.array([[[1.0, 0.0]], [[1.0, 0.0]]]), np.array([[[1.0, 0.0]], [[1.0, 0.0]]]),
                                     [1, 2], np.eye(2)[None])
    out = oracle_mod.decode_multi(q_abs.reshape(1, 2, 1, 2), q_rot.reshape(1, 2, 1, 2), vp, kp, np.array([[0]]),
                                  [3], G=1, d_n=2)
    assert abs(out[0, 0, 0, 0] - 0.674772102235) < 1e-7 and out[0, 0, 0, 1] == 0.0
    assert abs(out[0, 1, 0, 0] - 1.492296285352) < 1e-7


def test_multi_query_decode_is_causally_masked_attention(oracle_mod):
    # n_q queries on the last n_q positions == torch SDPA over the materialised keys
    # [v_j ; k_r,j] with the mask j <= T - n_q + i, one row per (query, head)
    n_q = 3
    w = synth.custom(dtype="bf16", B=2, H=4, G=2, d_v=32, d_r=16, T_range=(3, 150), shuffled=True)
    lens = torch.tensor([150, 70], dtype=torch.int32)
    inp, vp, kp = _rand_cache(w, seed=5, lens=lens)
    table = inp.block_table.numpy()
    g = torch.Generator().manual_seed(6)
    qa = torch.randn((2, n_q, 4, 32), generator=g, dtype=torch.float64).numpy()
    qr = torch.randn((2, n_q, 4, 16), generator=g, dtype=torch.float64).numpy()
    out = oracle_mod.decode_multi(qa, qr, vp, kp, table, lens.numpy(), G=2)
    for b in range(2):
        T = int(lens[b])
        for h in range(4):
            V = _gather_rows(vp, table, b, T, g=h // 2)
            KR = _gather_rows(kp, table, b, T)
            K = torch.tensor(np.concatenate([V, KR], axis=1))
            q = torch.tensor(np.concatenate([qa[b, :, h], qr[b, :, h]], axis=1))
            mask = torch.arange(T)[None, :] <= (T - n_q + torch.arange(n_q))[:, None]
            ref = F.scaled_dot_product_attention(q[None, None], K[None, None], torch.tensor(V)[None, None],
                                                 attn_mask=mask[None, None], scale=1 / math.sqrt(48))[0, 0]
            assert np.abs(out[b, :, h] - ref.numpy()).max() < 1e-12


def test_single_query_multi_decode_is_decode(oracle_mod):
    w = synth.custom(dtype="bf16", B=3, H=4, G=2, d_v=32, d_r=16, T_range=(1, 200), shuffled=True)
    inp, vp, kp = _rand_cache(w, seed=7)
    table, lens = inp.block_table.numpy(), inp.seq_lens.numpy()
    qa, qr = inp.q_abs.double().numpy(), inp.q_rot.double().numpy()
    one = oracle_mod.decode(qa, qr, vp, kp, table, lens, G=2)
    multi = oracle_mod.decode_multi(qa[:, None], qr[:, None], vp, kp, table, lens, G=2)
    assert np.array_equal(one, multi[:, 0])
    with pytest.raises(oracle_mod.OracleError):  # fewer context tokens than queries
        oracle_mod.decode_multi(np.zeros((3, 300, 4, 32)), np.zeros((3, 300, 4, 16)), vp, kp, table, lens, G=2)


# ---------------------------------------------------------------- special cases vs library

def _sdpa(q, k, v, scale):
    """torch fp64 attention of one query row against keys/values [T, d]."""
    q = torch.tensor(q, dtype=torch.float64)[None, None, None, :]
    k = torch.tensor(k, dtype=torch.float64)[None, None]
    v = torch.tensor(v, dtype=torch.float64)[None, None]
    return F.scaled_dot_product_attention(q, k, v, scale=scale)[0, 0, 0].numpy()


def _rand_cache(w, seed=0, lens=None):
    inp = synth.decode_inputs(w, seed=seed, lens=lens)
    return inp, synth.pool_bits(inp.v_pool), synth.pool_bits(inp.kr_pool)


def _gather_rows(pool_np, table, b, T, g=None):
    """Rows 0..T-1 of sequence b, read through the block table with numpy fancy indexing."""
    j = np.arange(T)
    blk = table[b, j // 64]
    if g is None:
        rows = pool_np[blk, j % 64]
    else:
        rows = pool_np[blk, g, j % 64]
    if rows.dtype == np.uint16:
        rows = bits_to_f(rows.reshape(-1)).reshape(rows.shape)
    return rows.astype(np.float64)


def test_shared_kv_special_case_is_plain_attention(oracle_mod):
    # Shared KV (K = V): M_h = I and no positional slice -> textbook attention over V
    w = synth.custom(dtype="bf16", B=2, H=4, G=2, d_v=32, d_r=0, T=200)
    inp, vp, kp = _rand_cache(w)
    table = inp.block_table.numpy()
    q_c = inp.q_abs.double().numpy()
    q_abs, q_rot = oracle_mod.absorb(q_c, np.zeros((2, 4, 0)), [199, 199], np.tile(np.eye(32), (4, 1, 1)))
    out = oracle_mod.decode(q_abs, q_rot, vp, kp, table, inp.seq_lens.numpy(), G=2)
    for b in range(2):
        for h in range(4):
            V = _gather_rows(vp, table, b, 200, g=h // 2)
            ref = _sdpa(q_c[b, h], V, V, 1 / math.sqrt(32))
            assert np.abs(out[b, h] - ref).max() < 1e-12


def test_head_to_group_map_and_positional_term(oracle_mod):
    # full decode vs attention over explicit keys [q'.v + q_r.k_r] built per head from group h // r
    w = synth.custom(dtype="bf16", B=2, H=8, G=2, d_v=32, d_r=16, T=130)
    inp, vp, kp = _rand_cache(w, seed=4)
    table = inp.block_table.numpy()
    qa, qr = inp.q_abs.double().numpy(), inp.q_rot.double().numpy()
    out = oracle_mod.decode(qa, qr, vp, kp, table, inp.seq_lens.numpy(), G=2)
    scale = 1 / math.sqrt(32 + 16)
    for b in range(2):
        KR = _gather_rows(kp, table, b, 130)
        for h in range(8):
            V = _gather_rows(vp, table, b, 130, g=h // 4)
            ref = _sdpa(np.concatenate([qa[b, h], qr[b, h]]), np.concatenate([V, KR], 1), V, scale)
            assert np.abs(out[b, h] - ref).max() < 1e-12
    # a wrong map (h mod G) gives a different answer on this input
    V_wrong = _gather_rows(vp, table, 0, 130, g=1 % 2)
    KR = _gather_rows(kp, table, 0, 130)
    wrong = _sdpa(np.concatenate([qa[0, 1], qr[0, 1]]), np.concatenate([V_wrong, KR], 1), V_wrong, scale)
    assert np.abs(out[0, 1] - wrong).max() > 1e-3


def test_absorbed_equals_unabsorbed_and_materialised_key(oracle_mod):
    w = synth.custom(dtype="bf16", B=2, H=4, G=2, d_v=16, d_n=24, d_r=8, T=70)
    lens = synth.seq_lens(w)
    table, nb = synth.block_table(w, lens)
    raw = synth.raw_inputs(w, lens, n_new=70, seed=5, pos_new=[0, 0])
    vp = np.zeros((nb, 2, 64, 16), dtype=np.uint16)
    kp = np.zeros((nb, 64, 8), dtype=np.uint16)
    oracle_mod.append(synth.pool_bits(raw.v_new), synth.pool_bits(raw.kr_new), raw.pos_new.numpy(),
                      table.numpy(), vp, kp)
    q_c, q_r, M = raw.q_c.double().numpy(), raw.q_r.double().numpy(), raw.M.double().numpy()
    pos_q = raw.pos_q.numpy()
    qa, qr = oracle_mod.absorb(q_c, q_r, pos_q, M)
    absorbed = oracle_mod.decode(qa, qr, vp, kp, table.numpy(), lens.numpy(), G=2, d_n=24)
    unabsorbed = oracle_mod.decode_unabsorbed(q_c, q_r, pos_q, M, vp, kp, table.numpy(), lens.numpy(), G=2)
    assert np.abs(absorbed - unabsorbed).max() < 1e-12
    # library check of the page's formula: K_h = V_g M_h (row form), full key [K_h ; k~_r]
    scale = 1 / math.sqrt(24 + 8)
    for b in range(2):
        KR = _gather_rows(kp, table.numpy(), b, 70)
        for h in range(4):
            V = _gather_rows(vp, table.numpy(), b, 70, g=h // 2)
            K = V @ M[h]
            qrot = oracle_mod.rope(q_r[b, h], pos_q[b])
            ref = _sdpa(np.concatenate([q_c[b, h], qrot]), np.concatenate([K, KR], 1), V, scale)
            assert np.abs(absorbed[b, h] - ref).max() < 1e-12
    # and the transposed map (q' = M^T q_c) is detectably wrong
    qa_t = np.einsum("hki,bhk->bhi", M.transpose(0, 2, 1), q_c) if M.shape[1] == M.shape[2] else None
    assert qa_t is None or np.abs(qa_t - qa).max() > 1e-3


def test_single_token_zero_query_and_constant_values(oracle_mod):
    w = synth.custom(dtype="f32", B=1, H=2, G=1, d_v=8, d_r=4, T=100)
    inp, vp, kp = _rand_cache(w, seed=6)
    table = inp.block_table.numpy()
    qa, qr = inp.q_abs.double().numpy(), inp.q_rot.double().numpy()
    # T = 1 -> o = v_0 exactly
    out = oracle_mod.decode(qa, qr, vp, kp, table, [1], G=1)
    assert np.array_equal(out[0, 0], vp[table[0, 0], 0, 0].astype(np.float64))
    # zero query -> uniform weights -> mean of the value rows
    out = oracle_mod.decode(np.zeros_like(qa), np.zeros_like(qr), vp, kp, table, [100], G=1)
    V = _gather_rows(vp, table, 0, 100, g=0)
    assert np.abs(out[0, 1] - V.mean(0)).max() < 1e-13
    # all value rows equal -> output is that row whatever the weights
    vc = vp.copy()
    vc[:] = np.float32(0.375)
    out = oracle_mod.decode(qa, qr, vc, kp, table, [100], G=1)
    assert np.abs(out - 0.375).max() < 1e-14


def test_split_invariance(oracle_mod):
    w = synth.custom(dtype="bf16", B=2, H=4, G=2, d_v=32, d_r=16, T=0, T_range=(70, 300))
    inp, vp, kp = _rand_cache(w, seed=7)
    table = inp.block_table.numpy()
    lens = inp.seq_lens.numpy()
    qa, qr = inp.q_abs.double().numpy(), inp.q_rot.double().numpy()
    for b in range(2):
        for h in range(4):
            ref = oracle_mod.decode_one(qa, qr, vp, kp, table, lens, G=2, b=b, h=h)
            for S in [1, 2, 3, 7, int(lens[b])]:
                got = oracle_mod.decode_split(qa, qr, vp, kp, table, lens, G=2, b=b, h=h, S=S)
                assert np.abs(got - ref).max() < 1e-12


def test_ragged_tail_ignores_slots_past_length(oracle_mod):
    w = synth.custom(dtype="bf16", B=1, H=2, G=1, d_v=16, d_r=8, T=77)
    inp, vp, kp = _rand_cache(w, seed=8)
    table = inp.block_table.numpy()
    qa, qr = inp.q_abs.double().numpy(), inp.q_rot.double().numpy()
    ref = oracle_mod.decode(qa, qr, vp, kp, table, [77], G=1)
    vp2, kp2 = vp.copy(), kp.copy()
    last = table[0, 1]
    vp2[last, :, 77 - 64:] = 0x7FC0  # NaN in every slot past the end
    kp2[last, 77 - 64:] = 0x7FC0
    got = oracle_mod.decode(qa, qr, vp2, kp2, table, [77], G=1)
    assert np.array_equal(got, ref)


def test_gqa_oracle_is_plain_attention(oracle_mod):
    w = synth.custom(dtype="bf16", B=2, H=4, G=2, d_v=32, d_r=0, T=150)
    inp = synth.decode_inputs(w, seed=9, k_pool=True)
    table = inp.block_table.numpy()
    kp, vp = synth.pool_bits(inp.extra["k_pool"]), synth.pool_bits(inp.v_pool)
    q = inp.extra["q"].double().numpy()
    for b in range(2):
        for h in range(4):
            got = oracle_mod.gqa_decode_one(q, kp, vp, table, inp.seq_lens.numpy(), G=2, b=b, h=h)
            K = _gather_rows(kp, table, b, 150, g=h // 2)
            V = _gather_rows(vp, table, b, 150, g=h // 2)
            assert np.abs(got - _sdpa(q[b, h], K, V, 1 / math.sqrt(32))).max() < 1e-12


# ---------------------------------------------------------------- paged layout and append

def test_layout_offsets_by_hand(oracle_mod):
    # G=4, d_v=64: block 2, group 3, slot 6, element 5 -> ((2*4+3)*64+6)*64+5
    assert oracle_mod.v_offset(4, 64, 2, 3, 6, 5) == ((2 * 4 + 3) * 64 + 6) * 64 + 5 == 45445
    assert oracle_mod.kr_offset(16, 2, 6, 5) == (2 * 64 + 6) * 16 + 5 == 2149


def test_append_is_a_bijection_onto_used_slots(oracle_mod):
    w = synth.custom(dtype="bf16", B=3, H=4, G=2, d_v=16, d_r=8, T=0, T_range=(10, 200), shuffled=True)
    lens = synth.seq_lens(w, seed_lens=3)
    table, nb = synth.block_table(w, lens, seed_lens=3, spare_blocks=2)
    n = int(lens.max())
    raw = synth.raw_inputs(w, lens, n_new=n, seed=10, pos_new=[0, 0, 0])
    sentinel = np.uint16(0xFFFF)  # a NaN pattern that no finite value takes
    vp = np.full((nb, 2, 64, 16), sentinel, dtype=np.uint16)
    kp = np.full((nb, 64, 8), sentinel, dtype=np.uint16)
    # per-sequence appends of exactly T_b tokens
    for b in range(3):
        T = int(lens[b])
        st = oracle_mod.append(synth.pool_bits(raw.v_new[b:b + 1, :T]), synth.pool_bits(raw.kr_new[b:b + 1, :T]),
                               [0], table[b:b + 1].numpy(), vp, kp)
        assert st == 0
    written = (vp != sentinel).reshape(nb, 2, 64, 16).all(axis=(1, 3))
    untouched = (vp == sentinel).reshape(nb, 2, 64, 16).all(axis=(1, 3))
    assert np.array_equal(written, ~untouched)   # slots are written whole or not at all
    assert written.sum() == int(lens.sum())     # one slot per token
    tb = table.numpy()
    for b in range(3):
        for p in [0, int(lens[b]) - 1, int(lens[b]) // 2]:
            blk, o = tb[b, p // 64], p % 64
            assert written[blk, o]
            assert np.array_equal(vp[blk, :, o], synth.pool_bits(raw.v_new[b, p]))  # bit copy
            want = oracle_mod.rope(bits_to_f(synth.pool_bits(raw.kr_new[b, p])), p)
            assert np.array_equal(kp[blk, o], np.array([oracle_mod.double_to_bf16(x) for x in want], np.uint16))
    # spare blocks stay untouched
    used = set(tb[tb >= 0].tolist())
    for blk in range(nb):
        if blk not in used:
            assert untouched[blk].all()


def test_append_rejects_positions_beyond_table(oracle_mod):
    w = synth.custom(dtype="f32", B=1, H=2, G=1, d_v=8, d_r=4, T=64)
    vp = np.zeros((1, 1, 64, 8), np.float32)
    kp = np.zeros((1, 64, 4), np.float32)
    st = oracle_mod.append(np.ones((1, 1, 1, 8), np.float32), np.ones((1, 1, 4), np.float32), [64],
                           np.array([[0]]), vp, kp, raise_on_index=False)
    assert st == 5 and not vp.any() and not kp.any()
    st = oracle_mod.append(np.ones((1, 1, 1, 8), np.float32), np.ones((1, 1, 4), np.float32), [3],
                           np.array([[7]]), vp, kp, raise_on_index=False)  # block id beyond the pool
    assert st == 5 and not vp.any()


def _golden_savings():
    rows = []
    with open(os.path.join(GOLDEN, "cache_saving.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                d_r, save, remain, exact = line.split()
                rows.append((int(d_r), int(save), int(remain), exact == "yes"))
    return rows


def test_cache_ratio_closed_form_matches_pages(oracle_mod):
    G, d_v = 4, 64
    for d_r, save, remain, exact in _golden_savings():
        ratio = oracle_mod.cache_ratio(G, d_v, d_r)
        assert ratio == (G * d_v + d_r) / (2 * G * d_v)
        if exact:
            assert ratio == 0.5
        assert round(100 * (1 - ratio)) == save and round(100 * ratio) == remain
    assert oracle_mod.cache_ratio(2, 32, 16) == 0.625
    assert oracle_mod.cache_ratio(8, 128, 24) == 0.51171875


def test_cache_ratio_equals_counted_pool_scalars(oracle_mod):
    # count the scalars one appended token occupies in the oracle's pools vs a K+V cache
    for G, d_v, d_r in [(4, 64, 16), (4, 64, 24), (8, 128, 24)]:
        vp = np.full((1, G, 64, d_v), 0xFFFF, np.uint16)
        kp = np.full((1, 64, d_r), 0xFFFF, np.uint16)
        oracle_mod.append(np.zeros((1, 1, G, d_v), np.uint16), np.zeros((1, 1, d_r), np.uint16), [5],
                          np.array([[0]]), vp, kp)
        used = int((vp != 0xFFFF).sum() + (kp != 0xFFFF).sum())
        gqa = 2 * G * d_v  # key and value rows for each of the G groups
        assert used / gqa == oracle_mod.cache_ratio(G, d_v, d_r)


# ---------------------------------------------------------------- fp8 (E4M3) value cache
#
# Not on the pages: the library's low-precision value cache.  E4M3 codes (OCP FP8: 4 exponent
# bits with bias 7, 3 mantissa bits, S.1111.111 = NaN, largest finite 448) with one
# power-of-two scale 2^e per (token, group); e is the smallest integer with
# max|v| <= 448 * 2^e (clamped to [-126, 120]); codes are v * 2^-e rounded once to nearest
# even, saturating at 448.  torch's float8_e4m3fn pins the format; closed forms pin the rest.

def e4m3_values_torch(codes):
    return torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def e4m3_codes_torch(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_on_every_code(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    want = e4m3_values_torch(codes)
    got = np.array([oracle_mod.e4m3_to_double(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(want)) and np.isnan(got).sum() == 2  # 0x7F, 0xFF
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e4m3_encode_matches_torch_in_range(oracle_mod):
    rng = np.random.default_rng(8)
    finite = e4m3_values_torch(np.arange(0, 0x7F, dtype=np.uint8))   # 0 .. 448, increasing
    mids = (finite[:-1] + finite[1:]) / 2                                # every tie, exact in fp32
    x = np.concatenate([rng.standard_normal(3000) * 40, rng.standard_normal(1000) * 2.0 ** -7,
                        mids, -mids, finite, -finite, rng.uniform(-463.9, 463.9, 1000)]).astype(np.float32)
    got = np.array([oracle_mod.double_to_e4m3(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, e4m3_codes_torch(x))


def test_e4m3_ties_saturation_and_specials(oracle_mod):
    enc = oracle_mod.double_to_e4m3
    assert enc(1.0) == 0x38 and enc(1.0625) == 0x38 and enc(1.1875) == 0x3A    # ties to the even code
    assert enc(2.0 ** -10) == 0x00 and enc(3 * 2.0 ** -11) == 0x01             # subnormal tie, round up
    assert enc(15 * 2.0 ** -10) == 0x08                                         # subnormal rounds to 2^-6
    assert enc(448.0) == 0x7E and enc(449.0) == 0x7E and enc(470.0) == 0x7E    # saturation, not NaN
    assert enc(1e30) == 0x7E and enc(-1e30) == 0xFE and enc(float("inf")) == 0x7E
    assert enc(float("nan")) == 0x7F and enc(0.0) == 0x00 and enc(-0.0) == 0x80


def test_fp8_exponent_closed_form(oracle_mod):
    e = oracle_mod.fp8_exponent
    assert e(448.0) == 0 and e(450.0) == 1 and e(1.0) == -8 and e(0.875) == -9 and e(0.0) == -126
    assert e(1e-40) == -126 and e(3.0e38) == 120
    rng = np.random.default_rng(9)
    for a in np.exp(rng.uniform(-80, 80, 2000)):
        k = e(float(a))
        assert 448.0 * 2.0 ** (k - 1) < a <= 448.0 * 2.0 ** k


def test_fp8_append_quantises_each_row(oracle_mod):
    """Each (token, group) row: the exponent from its largest magnitude, the codes torch's E4M3
    rounding of v * 2^-e; untouched slots keep their sentinel bytes; keys rotate as in bf16."""
    G, d_v, d_r, NB = 2, 64, 16, 3
    rng = np.random.default_rng(10)
    n = 70
    scale = np.exp(rng.uniform(-6, 6, (1, n, G, 1)))                 # rows of very different sizes
    v = (rng.standard_normal((1, n, G, d_v)) * scale).astype(np.float32)
    v[0, 3, 1] = 0.0                                                   # an all-zero row
    v_bits = bf16_bits(v)
    kr = bf16_bits(rng.standard_normal((1, n, d_r)))
    table = np.array([[2, 0]], np.int32)
    vp = np.full(NB * G * 64 * (d_v + 1), 0xA5, np.uint8)
    kp = np.full((NB, 64, d_r), 0xFFFF, np.uint16)
    assert oracle_mod.append(v_bits, kr, [0], table, vp, kp) == 0
    codes = vp[:NB * G * 64 * d_v].reshape(NB, G, 64, d_v)
    exps = vp[NB * G * 64 * d_v:].view(np.int8).reshape(NB, G, 64)
    vv = bits_to_f(v_bits)
    for t in range(n):
        blk, o = table[0, t // 64], t % 64
        for g in range(G):
            row = vv[0, t, g]
            amax = np.abs(row).max()
            k = -126 if amax == 0 else int(np.ceil(np.log2(amax / 448.0)))  # smallest k: amax <= 448 2^k
            assert exps[blk, g, o] == k
            assert oracle_mod.fp8_exp_offset(G, d_v, NB, blk, g, o) == NB * G * 64 * d_v + (blk * G + g) * 64 + o
            assert np.array_equal(codes[blk, g, o], e4m3_codes_torch(np.ldexp(row, -k)))
        # the positional key is the bf16 cache's: rotated at its position, rounded once
        want = np.array([oracle_mod.double_to_bf16(x) for x in oracle_mod.rope(bits_to_f(kr[0, t]), t)], np.uint16)
        assert np.array_equal(kp[blk, o], want)
    used_rows = {(table[0, t // 64], t % 64) for t in range(n)}
    for blk in range(NB):
        for o in range(64):
            if (blk, o) not in used_rows:
                assert (codes[blk, :, o] == 0xA5).all() and (exps[blk, :, o] == np.int8(-91)).all()
                assert (kp[blk, o] == 0xFFFF).all()


def test_fp8_round_trip_error_within_half_a_code(oracle_mod):
    """Dequantised values are within half an E4M3 spacing of the bf16 input, scaled by 2^e."""
    G, d_v, d_r = 1, 128, 2
    rng = np.random.default_rng(11)
    v = (rng.standard_normal((1, 64, G, d_v)) * np.exp(rng.uniform(-4, 4, (1, 64, G, 1)))).astype(np.float32)
    v_bits = bf16_bits(v)
    vp = np.zeros(G * 64 * (d_v + 1), np.uint8)
    kp = np.zeros((1, 64, d_r), np.uint16)
    oracle_mod.append(v_bits, bf16_bits(np.zeros((1, 64, d_r))), [0], np.array([[0]]), vp, kp)
    codes = vp[:64 * d_v].reshape(64, d_v)
    exps = vp[64 * d_v:].view(np.int8)
    x = bits_to_f(v_bits)[0, :, 0]
    deq = e4m3_values_torch(codes) * np.exp2(exps.astype(np.float64))[:, None]
    # spacing of E4M3 around |y| (y = x 2^-e): 2^(floor(log2|y|) - 3) for normals, 2^-9 below 2^-6
    y = np.abs(x) * np.exp2(-exps.astype(np.float64))[:, None]
    expo = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half = 0.5 * np.exp2(expo - 3) * np.exp2(exps.astype(np.float64))[:, None]
    assert (np.abs(deq - x) <= half).all()


def fp8_pool(rng, NB, G, d_v, emin=-12, emax=2):
    """Random fp8 value pool (no NaN codes) and the same values dequantised by torch into fp32."""
    codes = rng.integers(0, 256, (NB, G, 64, d_v)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] ^= 0x01                       # no NaN codes
    exps = rng.integers(emin, emax + 1, (NB, G, 64)).astype(np.int8)
    pool = np.concatenate([codes.reshape(-1), exps.view(np.uint8).reshape(-1)])
    vals = torch.ldexp(torch.tensor(codes).view(torch.float8_e4m3fn).double(),
                       torch.tensor(exps.astype(np.int64))[..., None].double())
    return pool, vals.float().numpy()


def test_fp8_decode_equals_decode_of_the_dequantised_values(oracle_mod):
    """Decode over the fp8 pool equals decode over an fp32 pool holding the values torch
    dequantises from the same codes and exponents (single-query, multi-query, unabsorbed)."""
    rng = np.random.default_rng(12)
    B, H, G, d_v, d_r = 3, 8, 2, 64, 16
    lens = np.array([1, 70, 130], np.int32)
    NB = 6
    table = np.array([[4, -1, -1], [0, 2, -1], [5, 1, 3]], np.int32)
    vp8, vp32 = fp8_pool(rng, NB, G, d_v)
    kp = bf16_bits(rng.standard_normal((NB, 64, d_r)))
    kp32 = bits_to_f(kp).astype(np.float32)
    qa = rng.standard_normal((B, H, d_v)) * 0.05
    qr = rng.standard_normal((B, H, d_r))
    got = oracle_mod.decode(qa, qr, vp8, kp, table, lens, G=G)
    want = oracle_mod.decode(qa, qr, vp32, kp32, table, lens, G=G)
    assert np.abs(got - want).max() <= 1e-12 * max(1.0, np.abs(want).max())
    qam = rng.standard_normal((B, 2, H, d_v)) * 0.05
    qrm = rng.standard_normal((B, 2, H, d_r))
    lens2 = np.maximum(lens, 2)
    got = oracle_mod.decode_multi(qam, qrm, vp8, kp, table, lens2, G=G)
    want = oracle_mod.decode_multi(qam, qrm, vp32, kp32, table, lens2, G=G)
    assert np.abs(got - want).max() <= 1e-12 * max(1.0, np.abs(want).max())
    q_c = rng.standard_normal((B, H, d_v))
    q_r = rng.standard_normal((B, H, d_r))
    M = rng.standard_normal((H, d_v, d_v)) / 8
    pos = lens - 1
    got = oracle_mod.decode_unabsorbed(q_c, q_r, pos, M, vp8, kp, table, lens, G=G)
    want = oracle_mod.decode_unabsorbed(q_c, q_r, pos, M, vp32, kp32, table, lens, G=G)
    assert np.abs(got - want).max() <= 1e-12 * max(1.0, np.abs(want).max())


def test_fp8_cache_bytes_per_token_counted_from_the_pools(oracle_mod):
    """Bytes one appended token occupies: G*d_v codes, G exponents and d_r bf16 key elements,
    against the bf16 cache and the matching bf16 K+V cache."""
    for G, d_v, d_r in [(4, 64, 16), (4, 64, 24), (8, 128, 24)]:
        vp = np.full(G * 64 * (d_v + 1), 0xA5, np.uint8)
        kp = np.full((1, 64, d_r), 0xFFFF, np.uint16)
        v = bf16_bits(np.full((1, 1, G, d_v), 0.75))          # exponent -9, code 0x7C (384)
        oracle_mod.append(v, bf16_bits(np.ones((1, 1, d_r))), [5], np.array([[0]]), vp, kp)
        codes, exps = vp[:G * 64 * d_v].reshape(G, 64, d_v), vp[G * 64 * d_v:].reshape(G, 64)
        used = int((codes[:, 5] != 0xA5).sum() + (exps[:, 5] != 0xA5).sum()) + 2 * int((kp[0, 5] != 0xFFFF).sum())
        assert used == G * d_v + G + 2 * d_r == oracle_mod.cache_bytes_per_token("fp8", G, d_v, d_r)
        assert oracle_mod.cache_bytes_per_token("bf16", G, d_v, d_r) == 2 * (G * d_v + d_r)
        gqa = 2 * (2 * G * d_v)
        assert (G * d_v + G + 2 * d_r) / gqa == pytest.approx((G * d_v + G + 2 * d_r) / (4 * G * d_v))
    # long-context layer: 292 bytes per token against 544 (bf16 GVA) and 1024 (bf16 GQA)
    assert oracle_mod.cache_bytes_per_token("fp8", 4, 64, 16) == 292
