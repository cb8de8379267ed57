"""The one-call decode step (gva_decode_step) on a B300.

The fused form forms the absorbed and rotated queries in the partial kernel's prologue and
appends the new token while the kernel streams the sequence's last block.  Its arithmetic is
the separate kernels' arithmetic in the same order, so each case checks:
  - output and both pools bit for bit against append + absorb + decode as three calls;
  - the output against the fp64 oracle (append, absorb, decode on the host copy of the cache)
    within the bf16 tolerances (max|d| <= 2e-2, relative RMS <= 5e-3).
Cases cover the kernel's instances (d_v 64/128, d_r 0..32, r = 1..8), the new token at the
first and the last row of a block, one-token contexts, and ranges that meet many segments.
"""
import dataclasses

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


def make_layer(w, **kw):
    return GVADecodeLayer(w.H, w.G, w.d_v, w.d_n, w.d_r, w.dtype, w.B, w.max_seq_len, **kw)


def assert_bf16_parity(got, want, what):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    d = np.abs(got - want)
    rrms = np.sqrt((d ** 2).mean()) / max(1e-30, np.sqrt((want ** 2).mean()))
    assert d.max() <= BF16_MAX and rrms <= BF16_RRMS, f"{what}: max|d| {d.max():.3e} rel rms {rrms:.3e}"


def run_both(w, seed, lens=None, mode=gva.GVA_STEP_FUSED):
    """Returns (inputs, raw step inputs, three-call output and pools, one-call output and pools)."""
    inp = synth.decode_inputs(w, seed=seed, device="cuda", lens=lens)
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=seed + 1, device="cuda")
    sep = make_layer(w)
    vp1, kp1 = inp.v_pool.clone(), inp.kr_pool.clone()
    out1 = sep.step(raw.q_c, raw.q_r, raw.pos_q, raw.M, raw.v_new, raw.kr_new, raw.pos_new, inp.block_table,
                    inp.seq_lens, vp1, kp1, overlap=False).clone()
    assert sep.device_error() == 0
    one = make_layer(w, step_mode=mode)
    vp2, kp2 = inp.v_pool.clone(), inp.kr_pool.clone()
    out2 = one.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, inp.seq_lens,
                          vp2, kp2).clone()
    assert one.device_error() == 0
    return inp, raw, (out1, vp1, kp1), (out2, vp2, kp2)


def oracle_step(w, inp, raw):
    """Host copy of the cache, the new token appended at T-1, the query absorbed at T-1, decoded."""
    vp = synth.pool_bits(inp.v_pool).copy()
    kp = synth.pool_bits(inp.kr_pool).copy()
    table = inp.block_table.cpu().numpy()
    lens = inp.seq_lens.cpu().numpy()
    oracle.append(synth.pool_bits(raw.v_new), synth.pool_bits(raw.kr_new), (lens - 1).astype(np.int32), table, vp, kp)
    qa, qr = oracle.absorb(raw.q_c.double().cpu().numpy(), raw.q_r.double().cpu().numpy(),
                           (lens - 1).astype(np.int32), raw.M.double().cpu().numpy())
    return oracle.decode(qa, qr, vp, kp, table, lens, G=w.G, d_n=w.d_n), vp, kp


STEP_CASES = [
    dict(B=5, H=16, G=4, d_v=64, d_r=16, T_range=(1, 3000)),    # long-context instance, ragged
    dict(B=4, H=32, G=8, d_v=128, d_r=24, T_range=(1, 2000)),   # ragged-batch instance
    dict(B=3, H=8, G=8, d_v=64, d_r=0, T_range=(60, 700)),      # r = 1, no positional slice
    dict(B=3, H=16, G=2, d_v=64, d_r=32, T_range=(1, 900)),     # r = 8, six warp pairs
    dict(B=6, H=16, G=4, d_v=128, d_r=8, T_range=(1, 400)),     # d_v = 128, one k8 step
    dict(B=4, H=8, G=4, d_v=64, d_r=24, T_range=(1, 200)),      # r = 2
]


@pytest.mark.parametrize("case", range(len(STEP_CASES)))
def test_fused_step_equals_three_calls_and_oracle(case):
    w = synth.custom(name=f"step{case}", dtype="bf16", shuffled=True, **STEP_CASES[case])
    inp, raw, (o1, v1, k1), (o2, v2, k2) = run_both(w, seed=200 + case)
    assert torch.equal(o1, o2), "fused output differs from the three calls"
    assert torch.equal(v1, v2) and torch.equal(k1, k2), "fused append differs from the append kernel"
    want, ovp, okp = oracle_step(w, inp, raw)
    assert_bf16_parity(o2.cpu().numpy(), want, f"case {case}")
    # the appended value rows are the new values bit for bit; nothing else moved
    assert np.array_equal(synth.pool_bits(v2), ovp)


@pytest.mark.parametrize("lens", [[64, 128, 1, 63, 65, 4096], [1, 1, 1, 1], [64 * 37] * 3])
def test_fused_step_block_edges(lens):
    """The new token on row 63 and row 0 of a block, one-token contexts, whole-block contexts."""
    w = synth.custom(name="edges", dtype="bf16", B=len(lens), H=16, G=4, d_v=64, d_r=16, T=max(lens),
                     shuffled=True)
    inp, raw, (o1, v1, k1), (o2, v2, k2) = run_both(w, seed=300, lens=lens)
    assert torch.equal(o1, o2) and torch.equal(v1, v2) and torch.equal(k1, k2)
    want, _, _ = oracle_step(w, inp, raw)
    assert_bf16_parity(o2.cpu().numpy(), want, f"lens {lens}")


def test_fused_step_many_segments_per_range():
    """Ranges that meet dozens of short sequences: the prologue forms the queries in batches."""
    w = synth.custom(name="many", dtype="bf16", B=700, H=16, G=4, d_v=64, d_r=16, T_range=(1, 300), shuffled=True)
    inp, raw, (o1, v1, k1), (o2, v2, k2) = run_both(w, seed=310)
    assert torch.equal(o1, o2) and torch.equal(v1, v2) and torch.equal(k1, k2)
    want, _, _ = oracle_step(w, inp, raw)
    assert_bf16_parity(o2.cpu().numpy(), want, "many segments")


@pytest.mark.parametrize("mode", [gva.GVA_STEP_AUTO, gva.GVA_STEP_SEPARATE])
def test_step_modes_agree(mode):
    w = synth.custom(name="modes", dtype="bf16", B=9, H=32, G=8, d_v=128, d_r=24, T_range=(1, 1500), shuffled=True)
    _, _, (o1, v1, k1), (o2, v2, k2) = run_both(w, seed=320, mode=mode)
    assert torch.equal(o1, o2) and torch.equal(v1, v2) and torch.equal(k1, k2)


def test_step_fp32_cache_runs_the_separate_kernels():
    """fp32 caches have no fused form: the one call runs the three kernels, and fused mode is
    rejected on the host."""
    w = synth.WORKLOADS[1]
    _, _, (o1, v1, k1), (o2, v2, k2) = run_both(w, seed=330, mode=gva.GVA_STEP_AUTO)
    assert torch.equal(o1, o2) and torch.equal(v1, v2) and torch.equal(k1, k2)
    layer = make_layer(w, step_mode=gva.GVA_STEP_FUSED)
    inp = synth.decode_inputs(w, seed=331, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=332, device="cuda")
    with pytest.raises(gva.GVAError) as e:
        layer.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, inp.seq_lens,
                         inp.v_pool, inp.kr_pool)
    assert e.value.status == gva.GVA_ERR_UNSUPPORTED


def test_fused_step_small_workspace_is_rejected():
    w = synth.custom(name="ws", dtype="bf16", B=3, H=16, G=4, d_v=64, d_r=16, T_range=(1, 500), shuffled=True)
    inp = synth.decode_inputs(w, seed=340, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=341, device="cuda")
    layer = make_layer(w, step_mode=gva.GVA_STEP_FUSED)
    need = gva.gva_decode_step_workspace_size(layer.ctx, w.B, w.max_seq_len)
    assert need > gva.gva_decode_workspace_size(layer.ctx, w.B, w.max_seq_len)
    small = torch.empty(gva.gva_decode_workspace_size(layer.ctx, w.B, w.max_seq_len), dtype=torch.uint8,
                        device="cuda")
    with pytest.raises(gva.GVAError) as e:
        gva.gva_decode_step(layer.ctx, raw.q_c, raw.q_r, raw.M, raw.v_new.reshape(w.B, w.G, w.d_v),
                            raw.kr_new.reshape(w.B, w.d_r), inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens,
                            w.max_seq_len, layer.out, small)
    assert e.value.status == gva.GVA_ERR_WORKSPACE


def test_fused_step_replays_in_a_cuda_graph():
    """The one-call step captured once and replayed gives the direct result (the append writes
    the same bits again)."""
    w = synth.custom(name="graph", dtype="bf16", B=4, H=16, G=4, d_v=64, d_r=16, T_range=(100, 900), shuffled=True)
    inp = synth.decode_inputs(w, seed=350, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=351, device="cuda")
    layer = make_layer(w, step_mode=gva.GVA_STEP_FUSED)

    def step():
        return layer.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, inp.seq_lens,
                                inp.v_pool, inp.kr_pool)
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


@pytest.mark.slow
@pytest.mark.parametrize("wid", [2, 3, 4])
def test_full_size_fused_step(wid):
    """The full-size workloads the automatic step mode fuses (350M layer, d_r = 24, long
    context), in the benchmark's launch configuration: one call against three, bit for bit, and
    every (b, h) row against the oracle's append + absorb + decode on a host copy of the cache."""
    w = synth.WORKLOADS[wid]
    inp, raw, (o1, v1, k1), (o2, v2, k2) = run_both(w, seed=0)
    assert torch.equal(o1, o2) and torch.equal(v1, v2) and torch.equal(k1, k2)
    del v1, k1, v2, k2
    want, _, _ = oracle_step(w, inp, raw)
    assert_bf16_parity(o2.cpu().numpy(), want, f"{w.name} fused step, all {w.B * w.H} rows")


def test_step_partial_then_combine_equals_one_call():
    """gva_decode_step (fused) is gva_decode_step_partial followed by gva_decode_combine."""
    w = synth.custom(name="passes", dtype="bf16", B=5, H=16, G=4, d_v=64, d_r=16, T_range=(1, 2500), shuffled=True)
    inp = synth.decode_inputs(w, seed=360, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=361, device="cuda")
    layer = make_layer(w, step_mode=gva.GVA_STEP_FUSED)
    v1, k1 = inp.v_pool.clone(), inp.kr_pool.clone()
    want = layer.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, inp.seq_lens,
                            v1, k1).clone()
    v2, k2 = inp.v_pool.clone(), inp.kr_pool.clone()
    layer.out.fill_(float("nan"))
    gva.gva_decode_step_partial(layer.ctx, raw.q_c, raw.q_r, raw.M, raw.v_new.reshape(w.B, w.G, w.d_v),
                                raw.kr_new.reshape(w.B, w.d_r), v2, k2, inp.block_table, inp.seq_lens, w.max_seq_len,
                                layer.workspace)
    gva.gva_decode_combine(layer.ctx, w.B, w.max_seq_len, layer.out, layer.workspace)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(layer.out, want) and torch.equal(v1, v2) and torch.equal(k1, k2)


def test_step_form_query():
    """gva_step_is_fused reports the form gva_decode_step takes."""
    few = synth.custom(name="few", dtype="bf16", B=8, H=16, G=4, d_v=64, d_r=16, T=4096)
    many = synth.custom(name="many", dtype="bf16", B=2048, H=16, G=4, d_v=64, d_r=16, T=256)
    lf, lm = make_layer(few), make_layer(many)
    assert gva.gva_step_is_fused(lf.ctx, few.B, few.max_seq_len) == 1
    assert gva.gva_step_is_fused(lm.ctx, many.B, many.max_seq_len) == 0
    gva.gva_set_step_mode(lm.ctx, gva.GVA_STEP_FUSED)
    assert gva.gva_step_is_fused(lm.ctx, many.B, many.max_seq_len) == 1
    gva.gva_set_step_mode(lf.ctx, gva.GVA_STEP_SEPARATE)
    assert gva.gva_step_is_fused(lf.ctx, few.B, few.max_seq_len) == 0
    f32 = make_layer(synth.WORKLOADS[1], step_mode=gva.GVA_STEP_FUSED)
    assert gva.gva_step_is_fused(f32.ctx, 1, 256) == -1
    gva.gva_set_step_mode(f32.ctx, gva.GVA_STEP_AUTO)
    assert gva.gva_step_is_fused(f32.ctx, 1, 256) == 0


@pytest.mark.parametrize("mode", [gva.GVA_STEP_FUSED, gva.GVA_STEP_SEPARATE])
def test_step_with_pinned_host_inputs_and_output(mode):
    """The step's inputs read from, and its output written to, pinned host memory give the bits of
    the step through device buffers."""
    w = synth.custom(name="pinned", dtype="bf16", B=5, H=16, G=4, d_v=64, d_r=16, T_range=(1, 1500), shuffled=True)
    inp = synth.decode_inputs(w, seed=370, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=371, device="cuda")
    layer = make_layer(w, step_mode=mode)
    v1, k1 = inp.v_pool.clone(), inp.kr_pool.clone()
    want = layer.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, inp.seq_lens,
                            v1, k1).clone()
    host = {k: getattr(raw, k).cpu().pin_memory() for k in ("q_c", "q_r", "v_new", "kr_new")}
    out = torch.full((w.B, w.H, w.d_v), float("nan")).pin_memory()
    v2, k2 = inp.v_pool.clone(), inp.kr_pool.clone()
    layer.fused_step(host["q_c"], host["q_r"], raw.M, host["v_new"], host["kr_new"], inp.block_table, inp.seq_lens,
                     v2, k2, out=out)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(out, want.cpu()) and torch.equal(v1, v2) and torch.equal(k1, k2)


def test_fused_step_bad_lengths_are_flagged_and_zeroed():
    """A length of 0 or past max_seq_len sets GVA_DEVERR_SEQ_LEN and zeroes that row; the other
    rows are unaffected, and the context stays usable."""
    w = synth.custom(name="badlen", dtype="bf16", B=4, H=16, G=4, d_v=64, d_r=16, T_range=(64, 300), shuffled=True)
    inp = synth.decode_inputs(w, seed=380, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=381, device="cuda")
    want, _, _ = oracle_step(w, inp, raw)
    lens = inp.seq_lens.clone()
    lens[1] = 0
    lens[2] = w.max_seq_len + 1
    layer = make_layer(w, step_mode=gva.GVA_STEP_FUSED)
    out = layer.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, lens,
                           inp.v_pool.clone(), inp.kr_pool.clone()).cpu().numpy()
    assert layer.device_error() & gva.GVA_DEVERR_SEQ_LEN
    assert np.all(out[1] == 0) and np.all(out[2] == 0)
    assert_bf16_parity(out[[0, 3]], want[[0, 3]], "rows beside bad lengths")
    layer.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, inp.seq_lens,
                     inp.v_pool.clone(), inp.kr_pool.clone())
    assert layer.device_error() == 0


def test_fused_step_bad_block_id_is_flagged():
    """A table entry outside the pool in a sequence's last block sets GVA_DEVERR_BLOCK_ID; that
    tile (and its append) is skipped, the other sequences are unaffected."""
    w = synth.custom(name="badblk", dtype="bf16", B=3, H=16, G=4, d_v=64, d_r=16, T_range=(100, 400), shuffled=True)
    inp = synth.decode_inputs(w, seed=385, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=386, device="cuda")
    want, _, _ = oracle_step(w, inp, raw)
    table = inp.block_table.clone()
    last = (int(inp.seq_lens[1]) - 1) // 64
    table[1, last] = inp.num_blocks + 5
    layer = make_layer(w, step_mode=gva.GVA_STEP_FUSED)
    out = layer.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, table, inp.seq_lens,
                           inp.v_pool.clone(), inp.kr_pool.clone()).cpu().numpy()
    assert layer.device_error() & gva.GVA_DEVERR_BLOCK_ID
    assert_bf16_parity(out[[0, 2]], want[[0, 2]], "rows beside a bad block id")


def test_fused_step_with_stale_nan_workspace():
    """Every stage the kernel reads is written in the same call: a workspace of NaN bytes gives the
    three calls' bits."""
    w = synth.custom(name="nanws", dtype="bf16", B=6, H=32, G=8, d_v=128, d_r=24, T_range=(1, 900), shuffled=True)
    inp = synth.decode_inputs(w, seed=390, device="cuda")
    raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=391, device="cuda")
    sep = make_layer(w)
    v1, k1 = inp.v_pool.clone(), inp.kr_pool.clone()
    want = sep.step(raw.q_c, raw.q_r, raw.pos_q, raw.M, raw.v_new, raw.kr_new, raw.pos_new, inp.block_table,
                    inp.seq_lens, v1, k1, overlap=False).clone()
    layer = make_layer(w, step_mode=gva.GVA_STEP_FUSED)
    layer.workspace.fill_(0xFF)
    v2, k2 = inp.v_pool.clone(), inp.kr_pool.clone()
    out = layer.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, inp.seq_lens, v2, k2)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(out, want) and torch.equal(v1, v2) and torch.equal(k1, k2)


def test_fused_step_largest_batch():
    """B = 8192: the lengths and the stages no longer fit beside the ring, so the prologue reads
    the lengths and keeps the stages in the workspace.  Bit for bit against the three calls,
    and against the oracle."""
    w = synth.custom(name="maxb", dtype="bf16", B=8192, H=16, G=4, d_v=64, d_r=16, T_range=(1, 200), shuffled=True)
    inp, raw, (o1, v1, k1), (o2, v2, k2) = run_both(w, seed=395)
    assert torch.equal(o1, o2) and torch.equal(v1, v2) and torch.equal(k1, k2)
    want, _, _ = oracle_step(w, inp, raw)
    assert_bf16_parity(o2.cpu().numpy(), want, "B=8192")


def test_fused_steps_on_two_streams():
    """Two contexts' fused steps issued on two streams at once give their results one by one."""
    wa = synth.custom(name="sa", dtype="bf16", B=6, H=16, G=4, d_v=64, d_r=16, T_range=(1, 3000), shuffled=True)
    wb = synth.custom(name="sb", dtype="bf16", B=4, H=32, G=8, d_v=128, d_r=24, T_range=(1, 2000), shuffled=True)
    runs = []
    for w, seed in ((wa, 400), (wb, 402)):
        inp = synth.decode_inputs(w, seed=seed, device="cuda")
        raw = synth.raw_inputs(w, inp.seq_lens.cpu(), n_new=1, seed=seed + 1, device="cuda")
        layer = make_layer(w, step_mode=gva.GVA_STEP_FUSED)
        runs.append((layer, inp, raw))

    def run(layer, inp, raw, stream=None):
        return layer.fused_step(raw.q_c, raw.q_r, raw.M, raw.v_new, raw.kr_new, inp.block_table, inp.seq_lens,
                                inp.v_pool, inp.kr_pool, stream=stream)
    want = [run(*r).clone() for r in runs]
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        for layer, _, _ in runs:
            layer.out.fill_(float("nan"))
        torch.cuda.synchronize()
        run(*runs[0], stream=sa)
        run(*runs[1], stream=sb)
        torch.cuda.synchronize()
        assert torch.equal(runs[0][0].out, want[0]) and torch.equal(runs[1][0].out, want[1])
    assert all(layer.device_error() == 0 for layer, _, _ in runs)


@pytest.mark.slow
@pytest.mark.parametrize("d_r", [0, 8, 32])
def test_full_size_fused_step_other_positional_widths(d_r):
    """The long-context workload at the other positional widths the kernel is built for (the
    d_r sweep: no positional slice, one k8 step, and the six-consumer instance of d_r = 32 with
    its patcher warp), full size: one call against three, bit for bit, and every (b, h) row
    against the oracle."""
    w = dataclasses.replace(synth.WORKLOADS[4], d_r=d_r, name=f"long-context-dr{d_r}")
    inp, raw, (o1, v1, k1), (o2, v2, k2) = run_both(w, seed=0)
    assert torch.equal(o1, o2) and torch.equal(v1, v2)
    if d_r:
        assert torch.equal(k1, k2)
    del v1, k1, v2, k2
    want, _, _ = oracle_step(w, inp, raw)
    assert_bf16_parity(o2.cpu().numpy(), want, f"{w.name} fused step, all {w.B * w.H} rows")
