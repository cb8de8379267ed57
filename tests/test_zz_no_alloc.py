"""gva_decode_attention_noalloc: decode attention for callers that cannot allocate device memory
(the library keeps its scratch in a fixed per-device array).  Its output must match the
workspace-taking gva_decode_attention on the same inputs bit for bit (same kernels, same split
plan), call after call, through the C ABI.
Kept in a file of its own that is collected last."""
import pytest
import torch

from compact_kv_cache_gva_b300 import gva, synth
from compact_kv_cache_gva_b300.layer import GVADecodeLayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


@pytest.mark.parametrize("wid,shape", [
    (1, None),
    (0, dict(dtype="bf16", B=6, H=16, G=4, d_v=64, d_r=16, T_range=(1, 2000), shuffled=True)),
    (0, dict(dtype="bf16", B=3, H=32, G=8, d_v=128, d_r=24, T_range=(64, 900), shuffled=True)),
])
def test_noalloc_matches_workspace_decode_on_consecutive_calls(wid, shape):
    w = synth.WORKLOADS[wid] if wid else synth.custom(**shape)
    layer = GVADecodeLayer(w.H, w.G, w.d_v, w.d_n, w.d_r, w.dtype, w.B, w.max_seq_len)
    assert gva.gva_decode_workspace_size(layer.ctx, w.B, w.max_seq_len) <= gva.NOALLOC_SCRATCH_BYTES
    # two calls in a row, on different inputs, each against the workspace-taking entry point
    for seed in (3, 4):
        inp = synth.decode_inputs(w, seed=seed, device="cuda")
        want = layer.attend(inp.v_pool, inp.kr_pool, inp.block_table, inp.seq_lens, q_abs=inp.q_abs,
                            q_rot=inp.q_rot).clone()
        out = torch.full_like(want, float("nan"))
        gva.gva_decode_attention_noalloc(layer.ctx, inp.q_abs, inp.q_rot if w.d_r else None, inp.v_pool,
                                         inp.kr_pool if w.d_r else None, inp.block_table, inp.seq_lens,
                                         w.max_seq_len, out)
        torch.cuda.synchronize()
        assert gva.gva_get_device_error(layer.ctx) == 0
        # same kernels, same split plan, same inputs: the same bits
        assert torch.equal(out, want)


def test_noalloc_rejects_batches_beyond_its_scratch():
    w = synth.custom(dtype="bf16", B=1024, H=32, G=8, d_v=128, d_r=24, T=64)
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_n, w.d_r, "bf16")
    assert gva.gva_decode_workspace_size(ctx, w.B, w.T) > gva.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((w.B, w.H, w.d_v), device="cuda")
    qr = torch.zeros((w.B, w.H, w.d_r), device="cuda")
    vp = torch.zeros((1, w.G, 64, w.d_v), dtype=torch.bfloat16, device="cuda")
    kp = torch.zeros((1, 64, w.d_r), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((w.B, 1), dtype=torch.int32, device="cuda")
    lens = torch.full((w.B,), 64, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(gva.GVAError) as e:
        gva.gva_decode_attention_noalloc(ctx, q, qr, vp, kp, table, lens, w.T, out)
    assert e.value.status == gva.GVA_ERR_WORKSPACE
