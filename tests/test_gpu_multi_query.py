"""Multi-query decode (n_q query tokens per sequence, the last n_q positions, causal) through
the C ABI, against the fp64 oracle.  Tolerances as for single-query bf16 decode."""
import math

import numpy as np
import pytest
import torch

import oracle
from compact_kv_cache_gva_b300 import gva, synth
from compact_kv_cache_gva_b300.layer import GVADecodeLayer

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_RRMS = 2e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    gva.load()


def assert_bf16(got, want, what):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape and np.isfinite(got).all(), what
    d = np.abs(got - want)
    rrms = math.sqrt((d ** 2).mean()) / math.sqrt((want ** 2).mean())
    assert d.max() <= BF16_MAX and rrms <= BF16_RRMS, f"{what}: max|d| {d.max():.3e} rel rms {rrms:.3e}"


def multi_inputs(w, n_q, seed, lens=None):
    inp = synth.decode_inputs(w, seed=seed, device="cuda", lens=lens)
    g = torch.Generator(device="cuda").manual_seed(seed + 100)
    qa = torch.randn((w.B, n_q, w.H, w.d_v), generator=g, device="cuda")
    qr = torch.randn((w.B, n_q, w.H, w.d_r), generator=g, device="cuda")
    return inp, qa, qr


def run_multi(w, inp, qa, qr, split_tokens=0):
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_n, w.d_r, "bf16")
    if split_tokens:
        gva.gva_set_split_tokens(ctx, split_tokens)
    n_q = qa.shape[1]
    ws = torch.empty(gva.gva_decode_workspace_size_multi(ctx, w.B, n_q, w.max_seq_len), dtype=torch.uint8,
                     device="cuda")
    out = torch.full((w.B, n_q, w.H, w.d_v), float("nan"), device="cuda")
    gva.gva_decode_attention_multi(ctx, qa, qr if w.d_r else None, inp.v_pool, inp.kr_pool if w.d_r else None,
                                   inp.block_table, inp.seq_lens, w.max_seq_len, out, ws)
    torch.cuda.synchronize()
    return out, ctx


def oracle_multi(w, inp, qa, qr):
    return oracle.decode_multi(qa.double().cpu().numpy(), qr.double().cpu().numpy(), synth.pool_bits(inp.v_pool),
                               synth.pool_bits(inp.kr_pool), inp.block_table.cpu().numpy(),
                               inp.seq_lens.cpu().numpy(), G=w.G, d_n=w.d_n)


CASES = [
    (dict(B=5, H=16, G=4, d_v=64, d_r=16, T_range=(2, 700)), 2, 0),      # R=4: one pass of 2
    (dict(B=4, H=16, G=4, d_v=64, d_r=24, T_range=(3, 900)), 3, 64 * 3),  # passes of 2 + 1
    (dict(B=3, H=8, G=4, d_v=64, d_r=16, T_range=(4, 500)), 4, 0),      # R=2: one pass of 4
    (dict(B=3, H=4, G=4, d_v=64, d_r=8, T_range=(5, 300)), 5, 64),       # R=1: passes of 4 + 1
    (dict(B=3, H=32, G=8, d_v=128, d_r=24, T_range=(2, 1200)), 2, 0),   # d_v = 128
    (dict(B=2, H=16, G=4, d_v=64, d_r=0, T_range=(2, 400)), 2, 0),       # no positional slice
    (dict(B=2, H=8, G=1, d_v=128, d_r=32, T_range=(8, 200)), 8, 0),      # R=8, d_v=128: 4 passes of 2 (16 pairs)
    (dict(B=4, H=16, G=4, d_v=64, d_r=16, T_range=(4, 3000)), 4, 0),     # R=4, d_v=64: one pass of 4
    (dict(B=3, H=16, G=4, d_v=64, d_r=24, T_range=(6, 900)), 6, 64 * 4),  # passes of 4 + 2
    (dict(B=3, H=16, G=2, d_v=64, d_r=16, T_range=(2, 700)), 2, 0),      # R=8, d_v=64: one pass of 2
    (dict(B=2, H=16, G=4, d_v=64, d_r=32, T_range=(4, 500)), 4, 0),      # d_r = 32, one pass of 4
    # prefill scale: sequence 0 is its queries alone (a whole causal prefill), the others decode
    # 128 (65) new tokens over a longer context
    (dict(B=3, H=16, G=4, d_v=64, d_r=16, T_range=(130, 700)), 128, 0),   # 32 passes of 4
    (dict(B=2, H=32, G=8, d_v=128, d_r=24, T_range=(66, 300)), 65, 0),    # d_v = 128: 16 passes of 4 + 1
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_multi_query_decode_matches_oracle(case):
    shape, n_q, split = CASES[case]
    w = synth.custom(dtype="bf16", shuffled=True, **shape)
    lens = synth.seq_lens(w, seed_lens=30 + case)
    lens[0] = n_q  # the shortest legal context: the queries are all there is
    lens[-1] = w.T_range[1]
    inp, qa, qr = multi_inputs(w, n_q, seed=40 + case, lens=lens)
    out, ctx = run_multi(w, inp, qa, qr, split_tokens=split)
    assert gva.gva_get_device_error(ctx) == 0
    assert_bf16(out.cpu().numpy(), oracle_multi(w, inp, qa, qr), f"case {case}")


def test_one_query_is_the_decode_call():
    w = synth.custom(dtype="bf16", B=6, H=16, G=4, d_v=64, d_r=16, T_range=(1, 900), shuffled=True)
    inp, qa, qr = multi_inputs(w, 1, seed=50)
    out, _ = run_multi(w, inp, qa, qr)
    layer = GVADecodeLayer(w.H, w.G, w.d_v, w.d_n, w.d_r, w.dtype, w.B, w.max_seq_len)
    want = layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=qa[:, 0].contiguous(),
                        q_rot=qr[:, 0].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0], want)


def test_context_shorter_than_the_queries_is_flagged_and_zeroed():
    w = synth.custom(dtype="bf16", B=3, H=16, G=4, d_v=64, d_r=16, T_range=(64, 300))
    lens = torch.tensor([200, 2, 300], dtype=torch.int32)
    inp, qa, qr = multi_inputs(w, 3, seed=60, lens=lens)
    out, ctx = run_multi(w, inp, qa, qr)
    assert gva.gva_get_device_error(ctx) & gva.GVA_DEVERR_SEQ_LEN
    got = out.cpu().numpy()
    assert np.all(got[1] == 0)
    inp.seq_lens[1] = 3
    want = oracle_multi(w, inp, qa, qr)
    assert_bf16(got[[0, 2]], want[[0, 2]], "other sequences unaffected")


def test_multi_query_needs_the_tensor_core_path():
    ctx = gva.gva_create(4, 2, 32, 32, 16, "f32")
    assert gva.gva_decode_workspace_size_multi(ctx, 1, 2, 256) == 0
    ctx = gva.gva_create(16, 4, 64, 64, 16, "bf16")
    gva.gva_set_decode_path(ctx, gva.GVA_PATH_FMA)
    assert gva.gva_decode_workspace_size_multi(ctx, 1, 2, 256) == 0
    assert gva.gva_decode_workspace_size_multi(ctx, 1, 1, 256) > 0


def test_speculative_step_from_raw_inputs():
    """Append n_q new tokens per sequence, absorb B*n_q query rows at their own positions, decode
    the n_q queries causally: both sides from the same raw draws."""
    n_q = 3
    w = synth.custom(dtype="bf16", B=3, H=16, G=4, d_v=64, d_r=16, T_range=(40, 600), shuffled=True)
    lens = synth.seq_lens(w, seed_lens=7)
    table, nb = synth.block_table(w, lens, seed_lens=7)
    T = int(lens.max())
    raw = synth.raw_inputs(w, lens, n_new=T, seed=70, pos_new=[0] * w.B)  # whole context as appended tokens
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_n, w.d_r, "bf16")
    vp = torch.zeros((nb, w.G, 64, w.d_v), dtype=torch.bfloat16, device="cuda")
    kp = torch.zeros((nb, 64, w.d_r), dtype=torch.bfloat16, device="cuda")
    tbl = table.cuda()
    for b in range(w.B):  # prefill all but the last n_q tokens, then append those n_q together
        Tb = int(lens[b])
        gva.gva_cache_append(ctx, raw.v_new[b:b + 1, :Tb - n_q].contiguous().cuda(),
                             raw.kr_new[b:b + 1, :Tb - n_q].contiguous().cuda(),
                             torch.zeros(1, dtype=torch.int32, device="cuda"), tbl[b:b + 1].contiguous(), vp, kp)
        gva.gva_cache_append(ctx, raw.v_new[b:b + 1, Tb - n_q:Tb].contiguous().cuda(),
                             raw.kr_new[b:b + 1, Tb - n_q:Tb].contiguous().cuda(),
                             torch.tensor([Tb - n_q], dtype=torch.int32, device="cuda"), tbl[b:b + 1].contiguous(),
                             vp, kp)
    g = torch.Generator().manual_seed(71)
    q_c = torch.randn((w.B * n_q, w.H, w.d_n), generator=g)
    q_r = torch.randn((w.B * n_q, w.H, w.d_r), generator=g)
    pos_q = (lens[:, None] - n_q + torch.arange(n_q)[None]).reshape(-1).to(torch.int32)
    q_abs = torch.empty((w.B * n_q, w.H, w.d_v), device="cuda")
    q_rot = torch.empty((w.B * n_q, w.H, w.d_r), device="cuda")
    gva.gva_absorb_query(ctx, q_c.cuda(), q_r.cuda(), pos_q.cuda(), raw.M.cuda(), q_abs, q_rot)
    ws = torch.empty(gva.gva_decode_workspace_size_multi(ctx, w.B, n_q, w.max_seq_len), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((w.B, n_q, w.H, w.d_v), device="cuda")
    gva.gva_decode_attention_multi(ctx, q_abs.view(w.B, n_q, w.H, w.d_v), q_rot.view(w.B, n_q, w.H, w.d_r), vp, kp,
                                   tbl, lens.cuda(), w.max_seq_len, out, ws)
    torch.cuda.synchronize()
    assert gva.gva_get_device_error(ctx) == 0
    ovp = np.zeros(vp.shape, np.uint16)
    okp = np.zeros(kp.shape, np.uint16)
    for b in range(w.B):
        Tb = int(lens[b])
        oracle.append(synth.pool_bits(raw.v_new[b:b + 1, :Tb]), synth.pool_bits(raw.kr_new[b:b + 1, :Tb]), [0],
                      table[b:b + 1].numpy(), ovp, okp)
    qa, qr = oracle.absorb(q_c.double().numpy(), q_r.double().numpy(), pos_q.numpy(), raw.M.double().numpy())
    want = oracle.decode_multi(qa.reshape(w.B, n_q, w.H, w.d_v), qr.reshape(w.B, n_q, w.H, w.d_r), ovp, okp,
                               table.numpy(), lens.numpy(), G=w.G, d_n=w.d_n)
    assert_bf16(out.cpu().numpy(), want, "speculative step")


STEP_CASES = [
    (dict(B=4, H=16, G=4, d_v=64, d_r=16, T_range=(3, 900)), 2),
    (dict(B=3, H=8, G=4, d_v=64, d_r=24, T_range=(4, 500)), 4),
    (dict(B=3, H=32, G=8, d_v=128, d_r=24, T_range=(3, 1200)), 3),
    (dict(B=2, H=16, G=4, d_v=64, d_r=0, T_range=(2, 400)), 2),
]


@pytest.mark.parametrize("case", range(len(STEP_CASES)))
def test_multi_query_one_call_step(case):
    """gva_decode_step_multi: append n_q tokens at the last n_q positions, absorb the n_q query
    rows there, decode -- bit for bit against the three calls, and against the oracle's append +
    absorb + multi-query decode on a host copy of the cache."""
    shape, n_q = STEP_CASES[case]
    w = synth.custom(name=f"mstep{case}", dtype="bf16", shuffled=True, **shape)
    lens = synth.seq_lens(w, seed_lens=60 + case)
    lens[0] = n_q
    inp = synth.decode_inputs(w, seed=70 + case, device="cuda", lens=lens)
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=n_q, seed=80 + case, device="cuda", n_q=n_q)
    mk = lambda: GVADecodeLayer(w.H, w.G, w.d_v, w.d_n, w.d_r, w.dtype, w.B, w.max_seq_len, n_q=n_q)
    sep, one = mk(), mk()
    v1, k1 = inp.v_pool.clone(), inp.kr_pool.clone()
    want = sep.step(raw.q_c, raw.q_r, raw.pos_q, raw.M, raw.v_new, raw.kr_new, raw.pos_new, inp.block_table,
                    inp.seq_lens, v1, k1, overlap=False).clone()
    v2, k2 = inp.v_pool.clone(), inp.kr_pool.clone()
    got = one.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, inp.seq_lens, v2, k2)
    torch.cuda.synchronize()
    assert sep.device_error() == 0 and one.device_error() == 0
    assert torch.equal(got, want) and torch.equal(v1, v2) and torch.equal(k1, k2)
    # the step's inputs read from, and its output written to, pinned host memory: same bits
    host = {k: getattr(raw, k).cpu().pin_memory() for k in ("q_c", "q_r", "v_new", "kr_new")}
    out_h = torch.full(tuple(want.shape), float("nan")).pin_memory()
    v3, k3 = inp.v_pool.clone(), inp.kr_pool.clone()
    one.fused_step(host["q_c"], host["q_r"], raw.M, host["v_new"], host["kr_new"], inp.block_table, inp.seq_lens,
                   v3, k3, out=out_h)
    torch.cuda.synchronize()
    assert one.device_error() == 0
    assert torch.equal(out_h, want.cpu()) and torch.equal(v3, v1) and torch.equal(k3, k1)
    # the oracle: append, absorb at T - n_q + i, causal multi-query decode
    vp, kp = synth.pool_bits(inp.v_pool).copy(), synth.pool_bits(inp.kr_pool).copy()
    table, L = inp.block_table.cpu().numpy(), inp.seq_lens.cpu().numpy()
    oracle.append(synth.pool_bits(raw.v_new), synth.pool_bits(raw.kr_new), (L - n_q).astype(np.int32), table, vp, kp)
    qa, qr = oracle.absorb(raw.q_c.double().cpu().numpy(), raw.q_r.double().cpu().numpy(),
                           raw.pos_q.cpu().numpy(), raw.M.double().cpu().numpy())
    want_o = oracle.decode_multi(qa.reshape(w.B, n_q, w.H, w.d_v), qr.reshape(w.B, n_q, w.H, w.d_r), vp, kp, table,
                                 L, G=w.G, d_n=w.d_n)
    assert_bf16(got.cpu().numpy(), want_o, f"one-call step, case {case}")


# ------------------------------------------------------------------------------- full-size workloads

@pytest.mark.slow
@pytest.mark.parametrize("n_q", [2, 4])
def test_full_size_long_context_multi_query_all_rows(n_q):
    """The long-context workload (570 MB of cache) with n_q queries per sequence, one pass in the
    launch configuration the benchmark times: every (b, query, h) row against the oracle, which
    reads a host copy of the whole cache."""
    w = synth.WORKLOADS[4]
    inp, qa, qr = multi_inputs(w, n_q, seed=40 + n_q)
    out, ctx = run_multi(w, inp, qa, qr)
    assert gva.gva_get_device_error(ctx) == 0
    assert_bf16(out.cpu().numpy(), oracle_multi(w, inp, qa, qr), f"long-context, n_q = {n_q}, all rows")


@pytest.mark.slow
def test_full_size_ragged_four_queries_all_rows():
    """The ragged paged batch (4.26 GB of cache, shuffled blocks, d_v = 128) with four queries per
    sequence in one pass (16 column pairs, the query operand in shared memory): every
    (b, query, h) row against the oracle."""
    w = synth.WORKLOADS[5]
    inp, qa, qr = multi_inputs(w, 4, seed=45)
    out, ctx = run_multi(w, inp, qa, qr)
    assert gva.gva_get_device_error(ctx) == 0
    assert_bf16(out.cpu().numpy(), oracle_multi(w, inp, qa, qr), "ragged batch, n_q = 4, all rows")
