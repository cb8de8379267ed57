"""The fp8 (E4M3) value cache on a B300, through the C ABI, against the fp64 oracle.

The cache stores each (token, group) value row as E4M3 codes times a power-of-two scale 2^e
(the exponent after all codes); positional keys stay bf16.  Checks:
  - append: codes and exponents bit for bit against the oracle's quantisation, keys within one
    bf16 ulp, untouched slots keep their sentinel bytes;
  - decode: the bf16 tolerances (max|d| <= 2e-2, relative RMS <= 5e-3) against the oracle,
    which dequantises the same bytes exactly, over every kernel instance family (d_v 64/128,
    d_r 0..32, H/G 1..8), ragged and shuffled, with garbage bytes past each context;
  - the one-call step: fused against the three calls bit for bit (output and both pools),
    and against the oracle's append + absorb + decode;
  - the long-context workload at full size, every output row.
"""
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
    yield
    torch.cuda.synchronize()


def assert_bf16(got, want, what):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape and np.isfinite(got).all(), f"{what}: shape or non-finite"
    d = np.abs(got - want)
    rrms = math.sqrt((d ** 2).mean()) / max(1e-30, math.sqrt((want ** 2).mean()))
    assert d.max() <= BF16_MAX and rrms <= BF16_RRMS, f"{what}: max|d| {d.max():.3e} rel rms {rrms:.3e}"


def make_layer(w, **kw):
    return GVADecodeLayer(w.H, w.G, w.d_v, w.d_n, w.d_r, w.dtype, w.B, w.max_seq_len, **kw)


def oracle_decode(w, inp):
    return oracle.decode(inp.q_abs.double().cpu().numpy(), inp.q_rot.double().cpu().numpy(),
                         synth.pool_bits(inp.v_pool), synth.pool_bits(inp.kr_pool), inp.block_table.cpu().numpy(),
                         inp.seq_lens.cpu().numpy(), G=w.G, d_n=w.d_n)


# ------------------------------------------------------------------------------- append

@pytest.mark.parametrize("shape", [
    dict(B=3, H=16, G=4, d_v=64, d_r=16, T_range=(1, 300)),
    dict(B=2, H=32, G=8, d_v=128, d_r=24, T_range=(65, 200)),
    dict(B=2, H=4, G=2, d_v=64, d_r=0, T_range=(10, 130)),
])
def test_fp8_append_matches_oracle_quantisation(shape):
    w = synth.custom(dtype="fp8", shuffled=True, **shape)
    lens = synth.seq_lens(w, seed_lens=2)
    table, nb = synth.block_table(w, lens, seed_lens=2, spare_blocks=3)
    n = int(lens.max())
    raw = synth.raw_inputs(w, lens, n_new=n, seed=11, pos_new=[0] * w.B)
    # rows of very different sizes (exponents from about -15 to +2), one all-zero row
    g = torch.Generator().manual_seed(5)
    size = torch.exp(torch.empty((w.B, n, w.G, 1)).uniform_(-6, 6, generator=g))
    v_new = (raw.v_new.float() * size).to(torch.bfloat16)
    v_new[0, 0, 0] = 0.0
    vp_h = np.full(nb * w.G * 64 * (w.d_v + 1), 0xA5, np.uint8)
    kp_h = np.full((nb, 64, w.d_r), 0xFFFF, np.uint16)
    vp_d = torch.from_numpy(vp_h.copy()).cuda()
    kp_d = torch.from_numpy(kp_h.view(np.int16).copy()).cuda().view(torch.bfloat16)
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_n, w.d_r, "fp8")
    tbl_d = table.cuda()
    for b in range(w.B):
        T = int(lens[b])
        vb, kb = v_new[b:b + 1, :T].contiguous(), raw.kr_new[b:b + 1, :T].contiguous()
        gva.gva_cache_append(ctx, vb.cuda(), kb.cuda(), torch.zeros(1, dtype=torch.int32, device="cuda"),
                             tbl_d[b:b + 1].contiguous(), vp_d, kp_d)
        assert oracle.append(synth.pool_bits(vb), synth.pool_bits(kb), [0], table[b:b + 1].numpy(), vp_h, kp_h) == 0
    torch.cuda.synchronize()
    assert gva.gva_get_device_error(ctx) == 0
    assert np.array_equal(vp_d.cpu().numpy(), vp_h), "codes and exponents must match the oracle bit for bit"
    gk = kp_d.view(torch.int16).cpu().numpy().view(np.uint16)
    a = gk.view(np.int16).astype(np.int64)
    bb = kp_h.view(np.int16).astype(np.int64)
    a = np.where(a < 0, -(a & 0x7FFF), a)
    bb = np.where(bb < 0, -(bb & 0x7FFF), bb)
    assert np.abs(a - bb).max(initial=0) <= 1
    assert np.array_equal(gk[kp_h == 0xFFFF], kp_h[kp_h == 0xFFFF])


# ------------------------------------------------------------------------------- decode

SHAPES = [
    dict(B=5, H=16, G=4, d_v=64, d_r=16, T_range=(1, 700)),
    dict(B=3, H=16, G=4, d_v=64, d_r=24, T_range=(60, 900)),
    dict(B=3, H=32, G=8, d_v=128, d_r=24, T_range=(100, 600)),
    dict(B=2, H=8, G=1, d_v=64, d_r=16, T_range=(1, 300)),    # R = 8
    dict(B=2, H=4, G=4, d_v=64, d_r=0, T_range=(5, 300)),     # R = 1, no positional slice
    dict(B=3, H=8, G=4, d_v=128, d_r=8, T_range=(1, 500)),    # R = 2, one k8 step
    dict(B=4, H=16, G=4, d_v=64, d_r=32, T_range=(1, 900)),   # d_r = 32
]


@pytest.mark.parametrize("split_tokens", [0, 64, 192])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_fp8_decode_matches_oracle(shape, split_tokens):
    w = synth.custom(dtype="fp8", shuffled=True, **SHAPES[shape])
    inp = synth.decode_inputs(w, seed=30 + shape, device="cuda", spare_blocks=2)
    layer = make_layer(w, split_tokens=split_tokens)
    out = layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=inp.q_abs, q_rot=inp.q_rot)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert_bf16(out.cpu().numpy(), oracle_decode(w, inp), f"fp8 shape {shape} split {split_tokens}")


def test_fp8_garbage_past_the_context_is_never_read():
    """Slots past each context hold NaN codes and out-of-range exponents: the output stays the
    oracle's (which never reads them)."""
    w = synth.custom(dtype="fp8", B=4, H=16, G=4, d_v=64, d_r=16, T_range=(1, 200), shuffled=True)
    inp = synth.decode_inputs(w, seed=33, device="cuda")
    want = oracle_decode(w, inp)
    codes, exps = gva.fp8_pool_views(inp.v_pool, w.G, w.d_v)
    for b in range(w.B):
        T = int(inp.seq_lens[b])
        last = int(inp.block_table[b, (T - 1) // 64])
        o = T % 64 if T % 64 else 64
        codes[last, :, o:] = 0x7F
        exps[last, :, o:] = 127 if b % 2 else -128
        inp.kr_pool[last, o:] = float("nan")
    layer = make_layer(w)
    out = layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=inp.q_abs, q_rot=inp.q_rot)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert_bf16(out.cpu().numpy(), want, "fp8 garbage tail")


def test_fp8_rejections():
    """The fp8 cache is read by single-query tensor-core decode only."""
    w = synth.custom(dtype="fp8", B=2, H=16, G=4, d_v=64, d_r=16, T=128)
    inp = synth.decode_inputs(w, seed=34, device="cuda")
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_n, w.d_r, "fp8")
    assert gva.gva_decode_workspace_size_multi(ctx, w.B, 2, w.max_seq_len) == 0
    with pytest.raises(gva.GVAError) as e:
        gva.gva_set_decode_path(ctx, gva.GVA_PATH_FMA)
        gva.gva_decode_plan(ctx, w.B, w.max_seq_len)
    assert e.value.status == gva.GVA_ERR_UNSUPPORTED
    with pytest.raises(gva.GVAError) as e:  # d_v = 32 has no tensor-core instance
        gva.gva_create(4, 2, 32, 32, 16, "fp8")
    assert e.value.status == gva.GVA_ERR_UNSUPPORTED
    # the comparison GQA kernel has no fp8 form: the library itself rejects the call
    ctx0 = gva.gva_create(w.H, w.G, w.d_v, w.d_n, 0, "fp8")
    out = torch.empty((w.B, w.H, w.d_v), device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    P = lambda t: gva.C.c_void_p(t.data_ptr())
    st = gva.load().gqa_decode_attention(ctx0.handle, w.B, P(inp.q_abs), P(inp.v_pool), P(inp.v_pool),
                                         P(inp.block_table), inp.block_table.shape[1], inp.num_blocks,
                                         P(inp.seq_lens), w.max_seq_len, P(out), P(ws), ws.numel(), gva._stream(None))
    assert st == gva.GVA_ERR_UNSUPPORTED


# ------------------------------------------------------------------------------- the one-call step

def run_step_both(w, seed, lens=None):
    inp = synth.decode_inputs(w, seed=seed, device="cuda", lens=lens)
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=seed + 1, device="cuda")
    sep = make_layer(w)
    vp1, kp1 = inp.v_pool.clone(), inp.kr_pool.clone()
    out1 = sep.step(raw.q_c, raw.q_r, raw.pos_q, raw.M, raw.v_new, raw.kr_new, raw.pos_new, inp.block_table,
                    inp.seq_lens, vp1, kp1, overlap=False).clone()
    assert sep.device_error() == 0
    one = make_layer(w, step_mode=gva.GVA_STEP_FUSED)
    vp2, kp2 = inp.v_pool.clone(), inp.kr_pool.clone()
    out2 = one.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, inp.seq_lens,
                          vp2, kp2).clone()
    assert one.device_error() == 0
    return inp, raw, (out1, vp1, kp1), (out2, vp2, kp2)


def oracle_step(w, inp, raw):
    vp = synth.pool_bits(inp.v_pool).copy()
    kp = synth.pool_bits(inp.kr_pool).copy()
    table = inp.block_table.cpu().numpy()
    lens = inp.seq_lens.cpu().numpy()
    oracle.append(synth.pool_bits(raw.v_new), synth.pool_bits(raw.kr_new), (lens - 1).astype(np.int32), table, vp, kp)
    qa, qr = oracle.absorb(raw.q_c.double().cpu().numpy(), raw.q_r.double().cpu().numpy(),
                           (lens - 1).astype(np.int32), raw.M.double().cpu().numpy())
    return oracle.decode(qa, qr, vp, kp, table, lens, G=w.G, d_n=w.d_n), vp, kp


STEP_SHAPES = [
    dict(B=5, H=16, G=4, d_v=64, d_r=16, T_range=(1, 3000)),
    dict(B=4, H=32, G=8, d_v=128, d_r=24, T_range=(1, 2000)),
    dict(B=3, H=8, G=8, d_v=64, d_r=0, T_range=(60, 700)),
    dict(B=3, H=16, G=2, d_v=64, d_r=32, T_range=(1, 900)),
]


@pytest.mark.parametrize("case", range(len(STEP_SHAPES)))
def test_fp8_fused_step_equals_three_calls_and_oracle(case):
    w = synth.custom(name=f"fp8step{case}", dtype="fp8", shuffled=True, **STEP_SHAPES[case])
    inp, raw, (o1, v1, k1), (o2, v2, k2) = run_step_both(w, seed=500 + case)
    assert torch.equal(v1, v2) and torch.equal(k1, k2), "the fused append's codes differ from the append kernel's"
    assert torch.equal(o1, o2), "fused output differs from the three calls"
    want, ovp, _ = oracle_step(w, inp, raw)
    assert np.array_equal(synth.pool_bits(v2), ovp), "the new token's codes and exponent differ from the oracle's"
    assert_bf16(o2.cpu().numpy(), want, f"fp8 step case {case}")


@pytest.mark.parametrize("lens", [[64, 128, 1, 63, 65], [1, 1, 1]])
def test_fp8_fused_step_block_edges(lens):
    w = synth.custom(name="fp8edges", dtype="fp8", B=len(lens), H=16, G=4, d_v=64, d_r=16, T=max(lens), shuffled=True)
    inp, raw, (o1, v1, k1), (o2, v2, k2) = run_step_both(w, seed=520, lens=lens)
    assert torch.equal(o1, o2) and torch.equal(v1, v2) and torch.equal(k1, k2)
    want, _, _ = oracle_step(w, inp, raw)
    assert_bf16(o2.cpu().numpy(), want, f"fp8 lens {lens}")


# ------------------------------------------------------------------------------- full size

@pytest.mark.slow
def test_fp8_long_context_full_size_all_rows():
    """The long-context layer over an fp8 value cache (292 bytes per token): the decode call and
    the fused step on every (b, h) row against the oracle; the step bit for bit against three calls."""
    w = synth.with_cache(synth.WORKLOADS[4], "fp8")
    inp = synth.decode_inputs(w, seed=0, device="cuda")
    layer = make_layer(w)
    out = layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=inp.q_abs, q_rot=inp.q_rot)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert_bf16(out.cpu().numpy(), oracle_decode(w, inp), "fp8 long-context decode, all rows")
    del layer
    inp, raw, (o1, v1, k1), (o2, v2, k2) = run_step_both(w, seed=0)
    assert torch.equal(o1, o2) and torch.equal(v1, v2) and torch.equal(k1, k2)
    del v1, k1, v2, k2
    want, _, _ = oracle_step(w, inp, raw)
    assert_bf16(o2.cpu().numpy(), want, "fp8 long-context fused step, all rows")


def test_fp8_cache_against_the_bf16_cache_of_the_same_values():
    """The same bf16 values appended to an fp8 and to a bf16 cache: the two decodes differ only by
    the quantisation (E4M3 keeps 3 mantissa bits); reported as a bound, not a parity claim."""
    wb = synth.custom(dtype="bf16", B=4, H=16, G=4, d_v=64, d_r=16, T=2048)
    wf = synth.with_cache(wb, "fp8")
    lens = synth.seq_lens(wb)
    table, nb = synth.block_table(wb, lens)
    raw = synth.raw_inputs(wb, lens, n_new=2048, seed=40, pos_new=[0] * wb.B, device="cuda")
    outs = []
    for w in (wb, wf):
        layer = make_layer(w)
        vp = (torch.zeros((nb, w.G, 64, w.d_v), dtype=torch.bfloat16, device="cuda") if w.dtype == "bf16" else
              torch.zeros(gva.fp8_value_pool_bytes(nb, w.G, w.d_v), dtype=torch.uint8, device="cuda"))
        kp = torch.zeros((nb, 64, w.d_r), dtype=torch.bfloat16, device="cuda")
        layer.append(raw.v_new, raw.kr_new, raw.pos_new, table.cuda(), vp, kp)
        layer.absorb(raw.q_c[:w.B], raw.q_r[:w.B], raw.pos_q[:w.B], raw.M)
        outs.append(layer.attend(vp, kp, table.cuda(), lens.cuda()).clone())
        assert layer.device_error() == 0
    d = (outs[1] - outs[0]).double()
    rel = (d.pow(2).mean().sqrt() / outs[0].double().pow(2).mean().sqrt()).item()
    assert rel < 0.05, f"fp8 against bf16 cache: relative RMS {rel:.3e}"


def test_fp8_step_form_query():
    """The automatic step mode fuses the fp8 step under the same rule as the bf16 one (small
    key maps, few segments per range); the separate mode still applies."""
    w = synth.custom(dtype="fp8", B=8, H=16, G=4, d_v=64, d_r=16, T=4096)
    layer = make_layer(w)
    assert gva.gva_step_is_fused(layer.ctx, w.B, w.max_seq_len) == 1
    gva.gva_set_step_mode(layer.ctx, gva.GVA_STEP_SEPARATE)
    assert gva.gva_step_is_fused(layer.ctx, w.B, w.max_seq_len) == 0
