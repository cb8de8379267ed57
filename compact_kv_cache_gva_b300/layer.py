"""One decode step of one GVA layer through the C ABI: absorb -> append -> decode, as three
calls (step) or as the library's one-call step (fused_step).

Holds the step's device buffers (absorbed/rotated queries, output, workspace) so a caller
only passes the step's inputs and the cache.  Marshalling only; the work is in libgva.so.
"""
import torch

from . import gva


class GVADecodeLayer:
    """With n_q > 1 a step decodes n_q query tokens per sequence (the last n_q positions, each
    reading the cache through its own position): query rows are b*n_q + i, out is [B,n_q,H,d_v]."""

    def __init__(self, H, G, d_v, d_n, d_r, cache_dtype, B, max_seq_len, device="cuda", split_tokens=0,
                 path=gva.GVA_PATH_AUTO, rope_base=10000.0, scale=0.0, n_q=1, step_mode=gva.GVA_STEP_AUTO):
        self.ctx = gva.gva_create(H, G, d_v, d_n, d_r, cache_dtype, rope_base, scale)
        if split_tokens:
            gva.gva_set_split_tokens(self.ctx, split_tokens)
        if path != gva.GVA_PATH_AUTO:
            gva.gva_set_decode_path(self.ctx, path)
        if step_mode != gva.GVA_STEP_AUTO:
            gva.gva_set_step_mode(self.ctx, step_mode)
        self.B, self.max_seq_len, self.n_q = B, max_seq_len, n_q
        self.q_abs = torch.empty((B * n_q, H, d_v), dtype=torch.float32, device=device)
        self.q_rot = torch.empty((B * n_q, H, d_r), dtype=torch.float32, device=device)
        self.out = torch.empty((B, H, d_v) if n_q == 1 else (B, n_q, H, d_v), dtype=torch.float32, device=device)
        ws = max(16, gva.gva_decode_workspace_size(self.ctx, B, max_seq_len) if n_q == 1 else
                 gva.gva_decode_workspace_size_multi(self.ctx, B, n_q, max_seq_len))
        ws = max(ws, gva.gva_decode_step_workspace_size_multi(self.ctx, B, n_q, max_seq_len))
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)
        self._side = None  # side stream of step(overlap=True), created on first use

    def plan(self):
        return gva.gva_decode_plan(self.ctx, self.B, self.max_seq_len)

    def absorb(self, q_c, q_r, pos_q, M, stream=None):
        gva.gva_absorb_query(self.ctx, q_c, q_r if self.ctx.dims.d_r else None, pos_q, M, self.q_abs,
                             self.q_rot if self.ctx.dims.d_r else None, stream)

    def append(self, v_new, kr_new, pos, block_table, v_pool, kr_pool, stream=None):
        gva.gva_cache_append(self.ctx, v_new, kr_new, pos, block_table, v_pool, kr_pool, stream)

    def attend(self, v_pool, kr_pool, block_table, seq_lens, q_abs=None, q_rot=None, stream=None):
        q_abs = self.q_abs if q_abs is None else q_abs
        q_rot = (self.q_rot if q_rot is None else q_rot) if self.ctx.dims.d_r else None
        kr_pool = kr_pool if self.ctx.dims.d_r else None
        if self.n_q == 1:
            gva.gva_decode_attention(self.ctx, q_abs, q_rot, v_pool, kr_pool, block_table, seq_lens,
                                     self.max_seq_len, self.out, self.workspace, stream)
        else:
            B, H = self.B, self.ctx.dims.H
            gva.gva_decode_attention_multi(self.ctx, q_abs.view(B, self.n_q, H, -1),
                                           None if q_rot is None else q_rot.view(B, self.n_q, H, -1), v_pool,
                                           kr_pool, block_table, seq_lens, self.max_seq_len, self.out,
                                           self.workspace, stream)
        return self.out

    def step(self, q_c, q_r, pos_q, M, v_new, kr_new, pos_new, block_table, seq_lens, v_pool, kr_pool, stream=None,
             overlap=True):
        """absorb the query, append the new token(s), attend through the current position.

        The append does not depend on the absorbed query, so with overlap=True it is issued on a
        side stream that forks from and joins back into the step's stream (also inside CUDA-graph
        capture), and the two small kernels run side by side."""
        main = torch.cuda.current_stream() if stream is None else stream
        if not overlap:
            self.absorb(q_c, q_r, pos_q, M, main)
            self.append(v_new, kr_new, pos_new, block_table, v_pool, kr_pool, main)
            return self.attend(v_pool, kr_pool, block_table, seq_lens, stream=main)
        if self._side is None:
            self._side = torch.cuda.Stream(device=main.device)
        self._side.wait_stream(main)
        self.append(v_new, kr_new, pos_new, block_table, v_pool, kr_pool, self._side)
        self.absorb(q_c, q_r, pos_q, M, main)
        main.wait_stream(self._side)
        return self.attend(v_pool, kr_pool, block_table, seq_lens, stream=main)

    def fused_step(self, q_c, q_r, M, v_new, kr_new, block_table, seq_lens, v_pool, kr_pool, stream=None,
                   out=None):
        """The whole step in one library call (gva_decode_step, or gva_decode_step_multi with
        n_q > 1): the new tokens (v_new [B,n_q,G,d_v], kr_new [B,n_q,d_r]; [B,G,d_v] and [B,d_r]
        also accepted when n_q == 1) go to the last n_q positions, which the lengths already
        count, and the query rows (q_c [B*n_q,H,d_n]) sit there.  The step's inputs and `out`
        (default: the layer's device buffer) may be pinned host tensors."""
        d = self.ctx.dims
        has_r = d.d_r > 0
        if self.n_q > 1:
            B, n = self.B, self.n_q
            gva.gva_decode_step_multi(self.ctx, q_c.reshape(B, n, d.H, d.d_n),
                                      q_r.reshape(B, n, d.H, d.d_r) if has_r else None, M,
                                      v_new.reshape(B, n, d.G, d.d_v), kr_new.reshape(B, n, d.d_r) if has_r else None,
                                      v_pool, kr_pool if has_r else None, block_table, seq_lens, self.max_seq_len,
                                      self.out if out is None else out, self.workspace, stream)
            return self.out if out is None else out
        gva.gva_decode_step(self.ctx, q_c, q_r if has_r else None, M, v_new.reshape(self.B, d.G, d.d_v),
                            kr_new.reshape(self.B, d.d_r) if has_r else None, v_pool, kr_pool if has_r else None,
                            block_table, seq_lens, self.max_seq_len, self.out if out is None else out, self.workspace,
                            stream)
        return self.out if out is None else out

    def device_error(self):
        return gva.gva_get_device_error(self.ctx)
