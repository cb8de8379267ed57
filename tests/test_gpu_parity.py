"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on a B300.

Tolerances: fp32 caches max|d| <= 1e-5; bf16 caches max|d| <= 2e-2 and relative RMS <= 5e-3,
both against the fp64 oracle on identical seeded inputs.  Cache appends: value rows bit for
bit, rotated positional keys within one unit in the last place of the cache dtype, every
untouched slot keeps its sentinel bits.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from compact_kv_cache_gva_b300 import gva, synth
from compact_kv_cache_gva_b300.layer import GVADecodeLayer

pytestmark = pytest.mark.gpu

F32_TOL = 1e-5
BF16_MAX, BF16_RRMS = 2e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    gva.load()
    yield
    torch.cuda.synchronize()


def assert_parity(got, want, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    d = np.abs(got - want)
    if dtype == "f32":
        assert d.max() <= F32_TOL, f"{what}: max|d| {d.max():.3e}"
    else:
        rrms = math.sqrt((d ** 2).mean()) / max(1e-30, math.sqrt((want ** 2).mean()))
        assert d.max() <= BF16_MAX and rrms <= BF16_RRMS, f"{what}: max|d| {d.max():.3e} rel rms {rrms:.3e}"
    return d.max()


def to_np_bits(t):
    return synth.pool_bits(t)


def ulp_distance(a_bits, b_bits, dtype):
    """Distance in units in the last place between two arrays of cache-dtype bit patterns."""
    if dtype == "f32":
        a = a_bits.view(np.int32).astype(np.int64)
        b = b_bits.view(np.int32).astype(np.int64)
        mask = 0x7FFFFFFF
    else:
        a = a_bits.view(np.int16).astype(np.int64)
        b = b_bits.view(np.int16).astype(np.int64)
        mask = 0x7FFF
    # map sign-magnitude to a monotone integer line
    a = np.where(a < 0, -(a & mask), a)
    b = np.where(b < 0, -(b & mask), b)
    return np.abs(a - b)


def make_layer(w, B=None, max_seq_len=None, **kw):
    return GVADecodeLayer(w.H, w.G, w.d_v, w.d_n, w.d_r, w.dtype, B or w.B, max_seq_len or w.max_seq_len, **kw)


def gather_sequence(inp, b, T=None):
    """Host copy of sequence b's blocks with an identity table (what the oracle reads for row b)."""
    T = int(inp.seq_lens[b]) if T is None else T
    nblk = (T + 63) // 64
    ids = inp.block_table[b, :nblk].long()
    vp = to_np_bits(inp.v_pool.index_select(0, ids))
    kp = to_np_bits(inp.kr_pool.index_select(0, ids))
    return vp, kp, np.arange(nblk, dtype=np.int32)[None], np.array([T], np.int32)


# ------------------------------------------------------------------------------- append

@pytest.mark.parametrize("dtype,shape", [
    ("f32", dict(B=1, H=4, G=2, d_v=32, d_r=16, T_range=(256, 256))),
    ("bf16", dict(B=4, H=16, G=4, d_v=64, d_r=16, T_range=(1, 300))),
    ("bf16", dict(B=3, H=32, G=8, d_v=128, d_r=24, T_range=(65, 200))),
])
def test_append_matches_oracle_layout(dtype, shape):
    w = synth.custom(dtype=dtype, shuffled=True, **shape)
    lens = synth.seq_lens(w, seed_lens=2)
    table, nb = synth.block_table(w, lens, seed_lens=2, spare_blocks=3)
    n = int(lens.max())
    raw = synth.raw_inputs(w, lens, n_new=n, seed=11, pos_new=[0] * w.B)
    sentinel = 0xFFFFFFFF if dtype == "f32" else 0xFFFF
    np_dt = np.uint32 if dtype == "f32" else np.uint16
    vp_h = np.full((nb, w.G, 64, w.d_v), sentinel, np_dt)
    kp_h = np.full((nb, 64, w.d_r), sentinel, np_dt)
    tdt = torch.int32 if dtype == "f32" else torch.int16
    vp_d = torch.from_numpy(vp_h.view(np.int32 if dtype == "f32" else np.int16).copy()).cuda().view(w.torch_dtype)
    kp_d = torch.from_numpy(kp_h.view(np.int32 if dtype == "f32" else np.int16).copy()).cuda().view(w.torch_dtype)
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_n, w.d_r, dtype)
    tbl_d = table.cuda()
    ov, ok = vp_h.view(np.float32) if dtype == "f32" else vp_h, kp_h.view(np.float32) if dtype == "f32" else kp_h
    for b in range(w.B):
        T = int(lens[b])
        v_new = raw.v_new[b:b + 1, :T].contiguous()
        kr_new = raw.kr_new[b:b + 1, :T].contiguous()
        gva.gva_cache_append(ctx, v_new.cuda(), kr_new.cuda(), torch.zeros(1, dtype=torch.int32, device="cuda"),
                             tbl_d[b:b + 1].contiguous(), vp_d, kp_d)
        assert oracle.append(to_np_bits(v_new), to_np_bits(kr_new), [0], table[b:b + 1].numpy(), ov, ok) == 0
    torch.cuda.synchronize()
    assert gva.gva_get_device_error(ctx) == 0
    gv = vp_d.view(tdt).cpu().numpy().view(np_dt)
    gk = kp_d.view(tdt).cpu().numpy().view(np_dt)
    assert np.array_equal(gv, vp_h), "value rows must be bit-exact and sentinels untouched"
    dist = ulp_distance(gk, kp_h, dtype)
    assert dist.max() <= 1, f"rotated key off by {dist.max()} ulp"
    untouched = kp_h == sentinel
    assert np.array_equal(gk[untouched], kp_h[untouched])
    # report how many rotated keys differ at all (expected: none or a handful of ties)
    assert (dist > 0).mean() < 1e-3


def test_append_skips_and_flags_unresolvable_slots():
    w = synth.custom(dtype="bf16", B=2, H=4, G=2, d_v=64, d_r=16, T_range=(10, 70))
    lens = torch.tensor([10, 70], dtype=torch.int32)
    table, nb = synth.block_table(w, lens)
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_n, w.d_r, "bf16")
    vp = torch.zeros((nb, 2, 64, 64), dtype=torch.bfloat16, device="cuda")
    kp = torch.zeros((nb, 64, 16), dtype=torch.bfloat16, device="cuda")
    raw = synth.raw_inputs(w, lens, n_new=1, seed=3)
    # sequence 0 has one block: position 64 has no table entry (-1)
    pos = torch.tensor([64, 5], dtype=torch.int32, device="cuda")
    gva.gva_cache_append(ctx, raw.v_new.cuda(), raw.kr_new.cuda(), pos, table.cuda(), vp, kp)
    bits = gva.gva_get_device_error(ctx)
    assert bits & gva.GVA_DEVERR_BLOCK_ID
    assert gva.gva_get_device_error(ctx) == 0  # read clears
    # sequence 1's token still landed (block table[1][0], slot 5)
    blk = int(table[1, 0])
    assert torch.equal(vp[blk, :, 5].cpu(), raw.v_new[1, 0])
    # a position past the table width is flagged as a position error
    pos = torch.tensor([2 * 64, 5], dtype=torch.int32, device="cuda")
    gva.gva_cache_append(ctx, raw.v_new.cuda(), raw.kr_new.cuda(), pos, table.cuda(), vp, kp)
    assert gva.gva_get_device_error(ctx) & gva.GVA_DEVERR_POSITION


# ------------------------------------------------------------------------------- absorb

@pytest.mark.parametrize("wid", [1, 2, 5])
def test_absorb_matches_oracle(wid):
    w = synth.WORKLOADS[wid]
    lens = synth.seq_lens(w)
    raw = synth.raw_inputs(w, lens, n_new=1, seed=12)
    layer = make_layer(w)
    layer.absorb(raw.q_c.cuda(), raw.q_r.cuda(), raw.pos_q.cuda(), raw.M.cuda())
    torch.cuda.synchronize()
    qa, qr = oracle.absorb(raw.q_c.double().numpy(), raw.q_r.double().numpy(), raw.pos_q.numpy(),
                           raw.M.double().numpy())
    ga, gr = layer.q_abs.cpu().double().numpy(), layer.q_rot.cpu().double().numpy()
    # the absorbed and rotated queries are fp32 results: the fp32 bound, absolute
    assert np.abs(ga - qa).max() <= F32_TOL
    assert np.abs(gr - qr).max() <= F32_TOL


def test_absorb_beyond_one_grid_of_row_blocks():
    """More query rows than one grid of 16-row blocks covers (65535 blocks in y): the kernel
    strides over the rest.  The last rows, and rows spread over the first grid, match the oracle."""
    ctx = gva.gva_create(1, 1, 32, 32, 2, "bf16")
    B = 65535 * 16 + 37
    g = torch.Generator(device="cuda").manual_seed(17)
    q_c = torch.randn((B, 1, 32), generator=g, device="cuda")
    q_r = torch.randn((B, 1, 2), generator=g, device="cuda")
    pos = torch.randint(0, 1 << 20, (B,), generator=g, device="cuda", dtype=torch.int32)
    M = torch.randn((1, 32, 32), generator=g, device="cuda") / math.sqrt(32)
    q_abs = torch.full((B, 1, 32), float("nan"), device="cuda")
    q_rot = torch.full((B, 1, 2), float("nan"), device="cuda")
    gva.gva_absorb_query(ctx, q_c, q_r, pos, M, q_abs, q_rot)
    torch.cuda.synchronize()
    assert gva.gva_get_device_error(ctx) == 0
    assert torch.isfinite(q_abs).all() and torch.isfinite(q_rot).all()
    rows = torch.cat([torch.arange(0, B, 4099), torch.arange(B - 700, B)]).to("cuda")
    qa, qr = oracle.absorb(q_c[rows].double().cpu().numpy(), q_r[rows].double().cpu().numpy(),
                           pos[rows].cpu().numpy(), M.double().cpu().numpy())
    assert np.abs(q_abs[rows].double().cpu().numpy() - qa).max() <= F32_TOL
    assert np.abs(q_rot[rows].double().cpu().numpy() - qr).max() <= F32_TOL


def test_step_rejects_pageable_host_buffers():
    """The one-call steps accept pinned host inputs and outputs, and reject pageable host memory
    before anything is enqueued: the cache is left untouched."""
    w = synth.custom(dtype="bf16", B=3, H=16, G=4, d_v=64, d_r=16, T_range=(10, 300), shuffled=True)
    inp = synth.decode_inputs(w, seed=55, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=2, seed=56, device="cuda", n_q=2)
    layer = make_layer(w, n_q=1)
    lib, st = gva.load(), gva._stream(None)
    paged_qc = np.zeros((w.B, w.H, w.d_n), np.float32)        # ordinary (pageable) host memory
    paged_out = np.zeros((w.B, w.H, w.d_v), np.float32)
    vp0, kp0 = inp.v_pool.clone(), inp.kr_pool.clone()
    P = lambda t: gva.C.c_void_p(t.data_ptr())
    common = (P(inp.v_pool), P(inp.kr_pool), P(inp.block_table), inp.block_table.shape[1], inp.num_blocks,
              P(inp.seq_lens), w.max_seq_len)
    qc_host = gva.C.c_void_p(paged_qc.ctypes.data)
    out_host = gva.C.c_void_p(paged_out.ctypes.data)
    v1, k1 = raw.v_new[:, 0].contiguous(), raw.kr_new[:, 0].contiguous()
    q_c1, q_r1 = raw.q_c[0::2].contiguous(), raw.q_r[0::2].contiguous()
    ws = P(layer.workspace), layer.workspace.numel()
    for qc, out in ((qc_host, P(layer.out)), (P(q_c1), out_host)):
        assert lib.gva_decode_step(layer.ctx.handle, w.B, qc, P(q_r1), P(raw.M), P(v1), P(k1), *common, out, *ws,
                                   st) == gva.GVA_ERR_INVALID_ARG
    assert lib.gva_decode_step_partial(layer.ctx.handle, w.B, qc_host, P(q_r1), P(raw.M), P(v1), P(k1), *common,
                                       *ws, st) == gva.GVA_ERR_INVALID_ARG
    multi = make_layer(w, n_q=2)
    wsm = P(multi.workspace), multi.workspace.numel()
    paged_qc2 = np.zeros((w.B, 2, w.H, w.d_n), np.float32)
    assert lib.gva_decode_step_multi(multi.ctx.handle, w.B, 2, gva.C.c_void_p(paged_qc2.ctypes.data), P(raw.q_r),
                                     P(raw.M), P(raw.v_new), P(raw.kr_new), *common, P(multi.out), *wsm,
                                     st) == gva.GVA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(inp.v_pool, vp0) and torch.equal(inp.kr_pool, kp0)
    assert layer.device_error() == 0


# ------------------------------------------------------------------------------- decode, small

def run_decode(w, inp, split_tokens=0, path=gva.GVA_PATH_AUTO, max_seq_len=None):
    layer = make_layer(w, max_seq_len=max_seq_len, split_tokens=split_tokens, path=path)
    out = layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=inp.q_abs, q_rot=inp.q_rot)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    return out.cpu().numpy(), layer


def oracle_decode_all(w, inp):
    return oracle.decode(inp.q_abs.double().cpu().numpy(), inp.q_rot.double().cpu().numpy(),
                         to_np_bits(inp.v_pool), to_np_bits(inp.kr_pool), inp.block_table.cpu().numpy(),
                         inp.seq_lens.cpu().numpy(), G=w.G, d_n=w.d_n)


@pytest.mark.parametrize("split_tokens", [0, 64, 128, 256])
def test_tiny_fp32_decode_matches_oracle(split_tokens):
    w = synth.WORKLOADS[1]
    inp = synth.decode_inputs(w, seed=0, device="cuda")
    got, layer = run_decode(w, inp, split_tokens=split_tokens)
    assert_parity(got, oracle_decode_all(w, inp), "f32", f"split {split_tokens}")


SMALL_BF16 = [
    dict(B=5, H=16, G=4, d_v=64, d_r=16, T_range=(1, 700)),
    dict(B=3, H=16, G=4, d_v=64, d_r=24, T_range=(60, 900)),
    dict(B=3, H=32, G=8, d_v=128, d_r=24, T_range=(100, 600)),
    dict(B=2, H=8, G=4, d_v=32, d_r=8, T_range=(1, 400)),
    dict(B=2, H=8, G=1, d_v=64, d_r=16, T_range=(1, 300)),   # r = 8
    dict(B=2, H=4, G=4, d_v=64, d_r=0, T_range=(5, 300)),    # r = 1, no positional slice
]


@pytest.mark.parametrize("path", [gva.GVA_PATH_FMA, gva.GVA_PATH_AUTO])
@pytest.mark.parametrize("split_tokens", [0, 64, 192])
@pytest.mark.parametrize("shape", range(len(SMALL_BF16)))
def test_small_bf16_decode_matches_oracle(shape, split_tokens, path):
    w = synth.custom(dtype="bf16", shuffled=True, **SMALL_BF16[shape])
    inp = synth.decode_inputs(w, seed=20 + shape, device="cuda", spare_blocks=2)
    got, _ = run_decode(w, inp, split_tokens=split_tokens, path=path)
    assert_parity(got, oracle_decode_all(w, inp), "bf16", f"shape {shape}")


# Shapes and split lengths that stress the tensor-core kernel's shared ring: few CTAs with
# long ranges (the ring wraps many times), many short sequences (segments shorter than the
# number of consumer warps, so warps skip whole segments), and ranges with fewer units than
# consumer warps.
RING_CASES = [
    (dict(B=16, H=16, G=4, d_v=64, d_r=16, T_range=(1, 3000)), 64 * 64),
    (dict(B=40, H=16, G=4, d_v=64, d_r=16, T_range=(1, 130)), 64 * 5),
    (dict(B=6, H=32, G=8, d_v=128, d_r=24, T_range=(1, 2500)), 64 * 48),
    (dict(B=3, H=8, G=1, d_v=128, d_r=32, T_range=(700, 1500)), 64 * 100),
    (dict(B=2, H=4, G=2, d_v=64, d_r=16, T_range=(1, 100)), 0),
    (dict(B=64, H=16, G=4, d_v=64, d_r=24, T_range=(1, 64)), 0),
    (dict(B=5, H=16, G=4, d_v=64, d_r=8, T_range=(1, 2000)), 0),      # trailing k8 step only
    (dict(B=4, H=16, G=4, d_v=128, d_r=0, T_range=(100, 1000)), 0),   # no positional slice
    (dict(B=6, H=16, G=4, d_v=64, d_r=32, T_range=(1, 3000)), 64 * 40),  # six warp pairs
]


@pytest.mark.parametrize("case", range(len(RING_CASES)))
def test_tensor_core_ring_schedules_match_oracle(case):
    shape, split = RING_CASES[case]
    w = synth.custom(dtype="bf16", shuffled=True, **shape)
    inp = synth.decode_inputs(w, seed=70 + case, device="cuda", spare_blocks=1)
    got, layer = run_decode(w, inp, split_tokens=split, path=gva.GVA_PATH_MMA)
    assert_parity(got, oracle_decode_all(w, inp), "bf16", f"ring case {case} plan {layer.plan()}")


@pytest.mark.parametrize("d", [64, 128])
def test_gqa_comparison_kernel_ring_depths(d):
    # at d = 128 the key and value tiles of a stage take 32 KB: the ring is shallower than the
    # number of consumer warps
    w = synth.custom(dtype="bf16", B=5, H=16, G=4, d_v=d, d_r=0, T_range=(1, 2000), shuffled=True)
    inp = synth.decode_inputs(w, seed=80 + d, device="cuda", k_pool=True)
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_v, 0, "bf16")
    gva.gva_set_split_tokens(ctx, 64 * 16)
    out = torch.empty((w.B, w.H, w.d_v), device="cuda")
    ws = torch.empty(gva.gva_decode_workspace_size(ctx, w.B, w.max_seq_len), dtype=torch.uint8, device="cuda")
    gva.gqa_decode_attention(ctx, inp.extra["q"], inp.extra["k_pool"], inp.v_pool, inp.block_table, inp.seq_lens,
                             w.max_seq_len, out, ws)
    torch.cuda.synchronize()
    assert gva.gva_get_device_error(ctx) == 0
    kp, vp = to_np_bits(inp.extra["k_pool"]), to_np_bits(inp.v_pool)
    q = inp.extra["q"].double().cpu().numpy()
    want = np.stack([np.stack([oracle.gqa_decode_one(q, kp, vp, inp.block_table.cpu().numpy(),
                                                     inp.seq_lens.cpu().numpy(), G=w.G, b=b, h=h)
                               for h in range(w.H)]) for b in range(w.B)])
    assert_parity(out.cpu().numpy(), want, "bf16", f"gqa d={d}")


def test_workspace_with_stale_nan_bytes():
    # the combine must never scale a record that holds no data (stale bytes may be NaN)
    w = synth.custom(dtype="bf16", B=9, H=16, G=4, d_v=64, d_r=16, T_range=(1, 300), shuffled=True)
    inp = synth.decode_inputs(w, seed=90, device="cuda")
    want = oracle_decode_all(w, inp)
    for path in (gva.GVA_PATH_FMA, gva.GVA_PATH_MMA):
        layer = make_layer(w, path=path)
        layer.workspace.fill_(0xFF)  # every float in the workspace is a NaN
        out = layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=inp.q_abs,
                           q_rot=inp.q_rot)
        torch.cuda.synchronize()
        assert layer.device_error() == 0
        assert_parity(out.cpu().numpy(), want, "bf16", f"stale workspace, path {path}")


@pytest.mark.parametrize("path", [gva.GVA_PATH_FMA, gva.GVA_PATH_AUTO])
def test_partial_then_combine_equals_one_call(path):
    """gva_decode_partial followed by gva_decode_combine gives gva_decode_attention's bits."""
    w = synth.custom(dtype="bf16", B=7, H=16, G=4, d_v=64, d_r=16, T_range=(1, 1500), shuffled=True)
    inp = synth.decode_inputs(w, seed=95, device="cuda")
    layer = make_layer(w, path=path)
    want = layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=inp.q_abs,
                        q_rot=inp.q_rot).clone()
    out = torch.full_like(want, float("nan"))
    gva.gva_decode_partial(layer.ctx, inp.q_abs, inp.q_rot, inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens,
                           w.max_seq_len, layer.workspace)
    gva.gva_decode_combine(layer.ctx, w.B, w.max_seq_len, out, layer.workspace)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(out, want)
    assert_parity(out.cpu().numpy(), oracle_decode_all(w, inp), "bf16", "two calls")


def test_ragged_tail_slots_are_never_read():
    # fill every slot past each sequence's end with NaN bits: the output must stay finite
    w = synth.custom(dtype="bf16", B=4, H=16, G=4, d_v=64, d_r=16, T_range=(1, 200), shuffled=True)
    inp = synth.decode_inputs(w, seed=31, device="cuda")
    want = oracle_decode_all(w, inp)
    for b in range(w.B):
        T = int(inp.seq_lens[b])
        last = int(inp.block_table[b, (T - 1) // 64])
        inp.v_pool[last, :, T % 64 if T % 64 else 64:] = float("nan")
        inp.kr_pool[last, T % 64 if T % 64 else 64:] = float("nan")
    for path in (gva.GVA_PATH_FMA, gva.GVA_PATH_AUTO):
        got, _ = run_decode(w, inp, path=path)
        assert_parity(got, want, "bf16", "nan tail")


def test_full_step_fp32_matches_oracle():
    """Raw inputs -> append (prefill of every token) + absorb + decode, both sides."""
    w = synth.WORKLOADS[1]
    lens = synth.seq_lens(w)
    table, nb = synth.block_table(w, lens)
    T = int(lens[0])
    raw = synth.raw_inputs(w, lens, n_new=T, seed=0, pos_new=[0])
    layer = make_layer(w)
    vp = torch.zeros((nb, w.G, 64, w.d_v), dtype=torch.float32, device="cuda")
    kp = torch.zeros((nb, 64, w.d_r), dtype=torch.float32, device="cuda")
    out = layer.step(raw.q_c.cuda(), raw.q_r.cuda(), raw.pos_q.cuda(), raw.M.cuda(), raw.v_new.cuda(),
                     raw.kr_new.cuda(), raw.pos_new.cuda(), table.cuda(), lens.cuda(), vp, kp).cpu().numpy()
    assert layer.device_error() == 0
    ovp = np.zeros((nb, w.G, 64, w.d_v), np.float32)
    okp = np.zeros((nb, 64, w.d_r), np.float32)
    oracle.append(raw.v_new.numpy(), raw.kr_new.numpy(), raw.pos_new.numpy(), table.numpy(), ovp, okp)
    qa, qr = oracle.absorb(raw.q_c.double().numpy(), raw.q_r.double().numpy(), raw.pos_q.numpy(),
                           raw.M.double().numpy())
    want = oracle.decode(qa, qr, ovp, okp, table.numpy(), lens.numpy(), G=w.G, d_n=w.d_n)
    assert_parity(out, want, "f32", "full step")
    # and against the unabsorbed form, which builds K_h = V_g M_h explicitly
    want_u = oracle.decode_unabsorbed(raw.q_c.double().numpy(), raw.q_r.double().numpy(), raw.pos_q.numpy(),
                                      raw.M.double().numpy(), ovp, okp, table.numpy(), lens.numpy(), G=w.G)
    assert_parity(out, want_u, "f32", "full step, unabsorbed oracle")


def test_gqa_comparison_kernel_matches_oracle():
    w = synth.custom(dtype="bf16", B=3, H=16, G=4, d_v=64, d_r=0, T_range=(1, 500), shuffled=True)
    inp = synth.decode_inputs(w, seed=40, device="cuda", k_pool=True)
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_v, 0, "bf16")
    out = torch.empty((w.B, w.H, w.d_v), device="cuda")
    ws = torch.empty(gva.gva_decode_workspace_size(ctx, w.B, w.max_seq_len), dtype=torch.uint8, device="cuda")
    gva.gqa_decode_attention(ctx, inp.extra["q"], inp.extra["k_pool"], inp.v_pool, inp.block_table, inp.seq_lens,
                             w.max_seq_len, out, ws)
    torch.cuda.synchronize()
    kp, vp = to_np_bits(inp.extra["k_pool"]), to_np_bits(inp.v_pool)
    q = inp.extra["q"].double().cpu().numpy()
    want = np.stack([np.stack([oracle.gqa_decode_one(q, kp, vp, inp.block_table.cpu().numpy(),
                                                     inp.seq_lens.cpu().numpy(), G=w.G, b=b, h=h)
                               for h in range(w.H)]) for b in range(w.B)])
    assert_parity(out.cpu().numpy(), want, "bf16", "gqa")


@pytest.mark.slow
def test_gqa_comparison_kernel_full_size_all_rows():
    """The same-build GQA decode at the size the benchmark times it beside GVA (the long-context
    shape over a 1.07 GB K+V cache): every (b, h) row against the oracle."""
    w4 = synth.WORKLOADS[4]
    w = synth.custom(name="long-context-gqa", dtype="bf16", B=w4.B, H=w4.H, G=w4.G, d_v=w4.d_v, d_r=0,
                     T=w4.T, T_range=w4.T_range, shuffled=w4.shuffled)
    inp = synth.decode_inputs(w, seed=1, device="cuda", k_pool=True)
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_v, 0, "bf16")
    out = torch.empty((w.B, w.H, w.d_v), device="cuda")
    ws = torch.empty(gva.gva_decode_workspace_size(ctx, w.B, w.max_seq_len), dtype=torch.uint8, device="cuda")
    gva.gqa_decode_attention(ctx, inp.extra["q"], inp.extra["k_pool"], inp.v_pool, inp.block_table, inp.seq_lens,
                             w.max_seq_len, out, ws)
    assert gva.gva_get_device_error(ctx) == 0
    kp, vp = to_np_bits(inp.extra["k_pool"]), to_np_bits(inp.v_pool)
    q = inp.extra["q"].double().cpu().numpy()
    table, lens = inp.block_table.cpu().numpy(), inp.seq_lens.cpu().numpy()
    want = np.stack([np.stack([oracle.gqa_decode_one(q, kp, vp, table, lens, G=w.G, b=b, h=h) for h in range(w.H)])
                     for b in range(w.B)])
    assert_parity(out.cpu().numpy(), want, "bf16", f"gqa, long-context shape, all {w.B * w.H} rows")


# ------------------------------------------------------------------------------- errors and edges

def test_host_side_errors():
    w = synth.custom(dtype="bf16", B=2, H=16, G=4, d_v=64, d_r=16, T_range=(64, 128))
    inp = synth.decode_inputs(w, seed=50, device="cuda")
    layer = make_layer(w)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gva.GVAError) as e:
        gva.gva_decode_attention(layer.ctx, inp.q_abs, inp.q_rot, inp.v_pool, inp.kr_pool, inp.block_table,
                                 inp.seq_lens, w.max_seq_len, layer.out, small)
    assert e.value.status == gva.GVA_ERR_WORKSPACE
    with pytest.raises(gva.GVAError) as e:  # table narrower than max_seq_len needs
        gva.gva_decode_attention(layer.ctx, inp.q_abs, inp.q_rot, inp.v_pool, inp.kr_pool,
                                 inp.block_table[:, :1].contiguous(), inp.seq_lens, w.max_seq_len, layer.out,
                                 layer.workspace)
    assert e.value.status == gva.GVA_ERR_INVALID_ARG
    with pytest.raises(gva.GVAError) as e:  # tensor-core path on an fp32 cache is unsupported
        ctx32 = gva.gva_create(4, 2, 32, 32, 16, "f32")
        gva.gva_set_decode_path(ctx32, gva.GVA_PATH_MMA)
        gva.gva_decode_plan(ctx32, 1, 256)
    assert e.value.status == gva.GVA_ERR_UNSUPPORTED
    # B == 0 is a no-op
    assert gva.load().gva_decode_attention(layer.ctx.handle, 0, None, None, None, None, None, 1, 1, None, 1,
                                           None, None, 0, None) == gva.GVA_OK


def test_bad_seq_len_is_flagged_and_zeroed():
    w = synth.custom(dtype="bf16", B=3, H=16, G=4, d_v=64, d_r=16, T_range=(64, 128))
    inp = synth.decode_inputs(w, seed=51, device="cuda")
    want = oracle_decode_all(w, inp)
    inp.seq_lens[1] = 0
    layer = make_layer(w)
    out = layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=inp.q_abs, q_rot=inp.q_rot)
    bits = layer.device_error()
    assert bits & gva.GVA_DEVERR_SEQ_LEN
    got = out.cpu().numpy()
    assert np.all(got[1] == 0)
    assert_parity(got[[0, 2]], want[[0, 2]], "bf16", "other rows unaffected")
    # the context stays usable
    inp.seq_lens[1] = 100
    layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=inp.q_abs, q_rot=inp.q_rot)
    assert layer.device_error() == 0


def test_single_token_context_returns_its_value():
    w = synth.custom(dtype="bf16", B=2, H=16, G=4, d_v=64, d_r=16, T_range=(1, 1))
    inp = synth.decode_inputs(w, seed=52, device="cuda")
    got, _ = run_decode(w, inp)
    for b in range(2):
        blk = int(inp.block_table[b, 0])
        for h in range(16):
            assert np.array_equal(got[b, h], inp.v_pool[blk, h // 4, 0].float().cpu().numpy())


# ------------------------------------------------------------------------------- full-size workloads

def sample_rows(w, inp, got, rows):
    qa = inp.q_abs.double().cpu().numpy()
    qr = inp.q_rot.double().cpu().numpy()
    want, have = [], []
    for b in sorted(set(b for b, _ in rows)):
        vp, kp, tb, sl = gather_sequence(inp, b)
        for bb, h in rows:
            if bb != b:
                continue
            want.append(oracle.decode_one(qa[b:b + 1], qr[b:b + 1], vp, kp, tb, sl, G=w.G, b=0, h=h, d_n=w.d_n))
            have.append(got[b, h])
    return np.array(have), np.array(want)


@pytest.mark.slow
@pytest.mark.parametrize("wid", [2, 3, 4, 5])
def test_full_size_workload_all_rows(wid):
    """Full-size cache in the launch configuration the benchmark uses: every (b, h) output row
    against the oracle (which reads a host copy of the whole cache, on all host cores)."""
    w = synth.WORKLOADS[wid]
    inp = synth.decode_inputs(w, seed=0, device="cuda")
    got, layer = run_decode(w, inp)
    assert_parity(got, oracle_decode_all(w, inp), "bf16", f"workload {wid}, all {w.B * w.H} rows")


@pytest.mark.parametrize("path", [gva.GVA_PATH_MMA, gva.GVA_PATH_FMA])
def test_largest_batch(path):
    """B = 8192 sequences, the library's batch limit: the prefix array takes 32 KB of shared
    memory beside the ring, and the combine merges 32768 segments.  Rows sampled for the oracle."""
    w = synth.custom(dtype="bf16", B=8192, H=16, G=4, d_v=64, d_r=16, T_range=(1, 200), shuffled=True)
    inp = synth.decode_inputs(w, seed=97, device="cuda")
    got, layer = run_decode(w, inp, path=path)
    rng = np.random.default_rng(97)
    lens = inp.seq_lens.cpu().numpy()
    bs = [0, w.B - 1, int(np.argmax(lens)), int(np.argmin(lens))] + list(rng.integers(0, w.B, 12))
    rows = [(int(b), int(h)) for b in bs for h in (0, int(rng.integers(0, w.H)), w.H - 1)]
    have, want = sample_rows(w, inp, got, rows)
    assert_parity(have, want, "bf16", f"B=8192 path {path}")
    assert np.isfinite(got).all()
    # one more sequence is rejected on the host, before anything is enqueued
    w2 = synth.custom(dtype="bf16", B=8193, H=16, G=4, d_v=64, d_r=16, T=64)
    inp2 = synth.decode_inputs(w2, seed=98, device="cuda")
    layer2 = make_layer(w2, path=path)
    assert gva.gva_decode_workspace_size(layer2.ctx, w2.B, w2.T) == 0
    with pytest.raises(gva.GVAError) as e:
        layer2.attend(inp2.v_pool, inp2.kr_pool, inp2.block_table, inp2.seq_lens, q_abs=inp2.q_abs,
                      q_rot=inp2.q_rot)
    assert e.value.status == gva.GVA_ERR_UNSUPPORTED


@pytest.mark.slow
def test_long_context_full_step_all_rows():
    """The three-call step on the long-context workload: absorb + append at T-1 + decode, every
    (b, h) row against the oracle's absorb + append + decode on a host copy of the cache."""
    w = synth.WORKLOADS[4]
    inp = synth.decode_inputs(w, seed=0, device="cuda")
    lens = inp.seq_lens
    raw = synth.raw_inputs(w, lens.cpu(), n_new=1, seed=7)
    vp, kp = to_np_bits(inp.v_pool).copy(), to_np_bits(inp.kr_pool).copy()
    layer = make_layer(w)
    out = layer.step(raw.q_c.cuda(), raw.q_r.cuda(), raw.pos_q.cuda(), raw.M.cuda(), raw.v_new.cuda(),
                     raw.kr_new.cuda(), raw.pos_new.cuda(), inp.block_table, lens, inp.v_pool, inp.kr_pool)
    got = out.cpu().numpy()
    assert layer.device_error() == 0
    table = inp.block_table.cpu().numpy()
    oracle.append(to_np_bits(raw.v_new), to_np_bits(raw.kr_new), raw.pos_new.numpy(), table, vp, kp)
    qa, qr = oracle.absorb(raw.q_c.double().numpy(), raw.q_r.double().numpy(), raw.pos_q.numpy(),
                           raw.M.double().numpy())
    want = oracle.decode(qa, qr, vp, kp, table, lens.cpu().numpy(), G=w.G, d_n=w.d_n)
    assert_parity(got, want, "bf16", "long-context step, all rows")


def test_step_replays_in_a_cuda_graph():
    """The three C-ABI calls of a step, captured once and replayed, give the direct result."""
    w = synth.custom(dtype="bf16", B=4, H=16, G=4, d_v=64, d_r=16, T_range=(100, 900), shuffled=True)
    inp = synth.decode_inputs(w, seed=60, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=61, device="cuda")
    layer = make_layer(w)

    def step():
        return layer.step(raw.q_c, raw.q_r, raw.pos_q, raw.M, raw.v_new, raw.kr_new, raw.pos_new, inp.block_table,
                          inp.seq_lens, inp.v_pool, inp.kr_pool)
    want = step().clone()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        step()
        cap.synchronize()
        with torch.cuda.graph(graph, stream=cap):
            step()
    torch.cuda.current_stream().wait_stream(cap)
    layer.out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(layer.out, want)


def test_two_streams_with_separate_workspaces():
    """Decodes of two contexts issued on two streams at once (each with its own workspace) give
    the results of running them one after the other."""
    wa = synth.custom(dtype="bf16", B=6, H=16, G=4, d_v=64, d_r=16, T_range=(1, 3000), shuffled=True)
    wb = synth.custom(dtype="bf16", B=4, H=32, G=8, d_v=128, d_r=24, T_range=(1, 2000), shuffled=True)
    ia, ib = synth.decode_inputs(wa, seed=101, device="cuda"), synth.decode_inputs(wb, seed=102, device="cuda")
    la, lb = make_layer(wa), make_layer(wb)

    def run(layer, inp, stream=None):
        return layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=inp.q_abs,
                            q_rot=inp.q_rot, stream=stream)
    want_a, want_b = run(la, ia).clone(), run(lb, ib).clone()
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        la.out.fill_(float("nan"))
        lb.out.fill_(float("nan"))
        torch.cuda.synchronize()
        run(la, ia, sa)
        run(lb, ib, sb)
        torch.cuda.synchronize()
        assert torch.equal(la.out, want_a) and torch.equal(lb.out, want_b)
    assert la.device_error() == 0 and lb.device_error() == 0


def test_multi_query_step_replays_in_a_cuda_graph():
    """A step with 2 query tokens per sequence (append 2 + absorb 2B rows + multi-query decode),
    captured once and replayed, gives the direct result."""
    w = synth.custom(dtype="bf16", B=4, H=16, G=4, d_v=64, d_r=16, T_range=(100, 900), shuffled=True)
    inp = synth.decode_inputs(w, seed=103, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=2, seed=104, device="cuda", n_q=2)
    layer = make_layer(w, n_q=2)

    def step():
        return layer.step(raw.q_c, raw.q_r, raw.pos_q, raw.M, raw.v_new, raw.kr_new, raw.pos_new, inp.block_table,
                          inp.seq_lens, inp.v_pool, inp.kr_pool)
    want = step().clone()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        step()
        cap.synchronize()
        with torch.cuda.graph(graph, stream=cap):
            step()
    torch.cuda.current_stream().wait_stream(cap)
    layer.out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(layer.out, want)
