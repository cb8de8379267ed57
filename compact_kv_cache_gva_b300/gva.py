"""Thin Python binding of libgva.so (the C ABI in include/gva.h), by ctypes.

Argument marshalling only: every function takes torch tensors, checks that they are CUDA,
contiguous and of the dtype the C ABI states, derives the sizes from their shapes, and
calls the C function of the same name on the current torch stream (or the stream given).
All computation happens in the library's kernels.  There is no CPU fallback: if the
library is missing or cannot be loaded, the first call raises.
"""
import ctypes as C
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgva.so")

GVA_OK, GVA_ERR_INVALID_ARG, GVA_ERR_UNSUPPORTED, GVA_ERR_WORKSPACE, GVA_ERR_CUDA, GVA_ERR_DEVICE_INDEX = range(6)
GVA_F32, GVA_BF16, GVA_FP8_E4M3 = 0, 1, 2
GVA_PATH_AUTO, GVA_PATH_FMA, GVA_PATH_MMA = 0, 1, 2
GVA_STEP_AUTO, GVA_STEP_FUSED, GVA_STEP_SEPARATE = 0, 1, 2
GVA_DEVERR_POSITION, GVA_DEVERR_BLOCK_ID, GVA_DEVERR_SEQ_LEN, GVA_DEVERR_TIMEOUT = 1, 2, 4, 8
BLOCK_TOKENS = 64

# Exported symbols the header declares (checked by the CPU tests).
EXPORTS = ("gva_create", "gva_destroy", "gva_absorb_query", "gva_cache_append", "gva_decode_workspace_size",
           "gva_decode_attention", "gqa_decode_attention", "gva_set_split_tokens", "gva_set_decode_path",
           "gva_decode_plan", "gva_get_device_error", "gva_status_string", "gva_version",
           "gva_decode_attention_noalloc", "gva_decode_partial", "gva_decode_combine",
           "gva_decode_attention_multi", "gva_decode_workspace_size_multi", "gva_decode_step",
           "gva_decode_step_workspace_size", "gva_set_step_mode", "gva_step_is_fused", "gva_decode_step_partial",
           "gva_decode_step_multi", "gva_decode_step_workspace_size_multi")
NOALLOC_SCRATCH_BYTES = 4 << 20


class GVAError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class gva_dims(C.Structure):
    _fields_ = [("H", C.c_int), ("G", C.c_int), ("d_v", C.c_int), ("d_n", C.c_int), ("d_r", C.c_int),
                ("block_size", C.c_int), ("cache_dtype", C.c_int), ("rope_base", C.c_double), ("scale", C.c_float)]


_lib = None


def load():
    """Loads libgva.so once; raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libgva.so is not built ({LIB_PATH}); run `python -m compact_kv_cache_gva_b300.build`")
    L = C.CDLL(LIB_PATH)
    vp, ip, i, st = C.c_void_p, C.c_void_p, C.c_int, C.c_void_p
    L.gva_create.argtypes = [C.POINTER(gva_dims), C.POINTER(C.c_void_p)]
    L.gva_destroy.argtypes = [vp]
    L.gva_destroy.restype = None
    L.gva_absorb_query.argtypes = [vp, i, vp, vp, ip, vp, vp, vp, st]
    L.gva_cache_append.argtypes = [vp, i, i, vp, vp, ip, ip, i, i, vp, vp, st]
    L.gva_decode_workspace_size.argtypes = [vp, i, i]
    L.gva_decode_workspace_size.restype = C.c_size_t
    L.gva_decode_attention.argtypes = [vp, i, vp, vp, vp, vp, ip, i, i, ip, i, vp, vp, C.c_size_t, st]
    L.gqa_decode_attention.argtypes = [vp, i, vp, vp, vp, ip, i, i, ip, i, vp, vp, C.c_size_t, st]
    L.gva_decode_attention_noalloc.argtypes = [vp, i, vp, vp, vp, vp, ip, i, i, ip, i, vp, st]
    L.gva_decode_partial.argtypes = [vp, i, vp, vp, vp, vp, ip, i, i, ip, i, vp, C.c_size_t, st]
    L.gva_decode_combine.argtypes = [vp, i, i, vp, vp, C.c_size_t, st]
    L.gva_decode_attention_multi.argtypes = [vp, i, i, vp, vp, vp, vp, ip, i, i, ip, i, vp, vp, C.c_size_t, st]
    L.gva_decode_workspace_size_multi.argtypes = [vp, i, i, i]
    L.gva_decode_workspace_size_multi.restype = C.c_size_t
    L.gva_decode_step.argtypes = [vp, i, vp, vp, vp, vp, vp, vp, vp, ip, i, i, ip, i, vp, vp, C.c_size_t, st]
    L.gva_decode_step_workspace_size.argtypes = [vp, i, i]
    L.gva_decode_step_workspace_size.restype = C.c_size_t
    L.gva_set_step_mode.argtypes = [vp, i]
    L.gva_step_is_fused.argtypes = [vp, i, i]
    L.gva_decode_step_multi.argtypes = [vp, i, i, vp, vp, vp, vp, vp, vp, vp, ip, i, i, ip, i, vp, vp, C.c_size_t, st]
    L.gva_decode_step_workspace_size_multi.argtypes = [vp, i, i, i]
    L.gva_decode_step_workspace_size_multi.restype = C.c_size_t
    L.gva_decode_step_partial.argtypes = [vp, i, vp, vp, vp, vp, vp, vp, vp, ip, i, i, ip, i, vp, C.c_size_t, st]
    L.gva_set_split_tokens.argtypes = [vp, i]
    L.gva_set_decode_path.argtypes = [vp, i]
    L.gva_decode_plan.argtypes = [vp, i, i, C.POINTER(C.c_int), C.POINTER(C.c_int)]
    L.gva_get_device_error.argtypes = [vp, C.POINTER(C.c_uint)]
    L.gva_status_string.argtypes = [i]
    L.gva_status_string.restype = C.c_char_p
    L.gva_version.argtypes = []
    L.gva_step_is_fused.restype = C.c_int
    for name in EXPORTS:
        if name not in ("gva_destroy", "gva_decode_workspace_size", "gva_decode_workspace_size_multi",
                        "gva_decode_step_workspace_size", "gva_decode_step_workspace_size_multi",
                        "gva_status_string", "gva_version", "gva_step_is_fused"):
            getattr(L, name).restype = C.c_int
    _lib = L
    return L


def status_string(status):
    try:
        return load().gva_status_string(int(status)).decode()
    except Exception:
        return "unknown"


def _check(status, what):
    if status != GVA_OK:
        raise GVAError(status, what)


def _stream(stream):
    if stream is None:
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _ptr(t, dtype, name, allow_none=False, allow_pinned=False):
    """Pointer of a CUDA tensor (or, with allow_pinned, of a pinned host tensor, which the
    kernels read or write directly through its mapped address)."""
    if t is None:
        if allow_none:
            return C.c_void_p(0)
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not (t.is_cuda or (allow_pinned and t.is_pinned())):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if allow_pinned else ""))
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return C.c_void_p(t.data_ptr())


class Context:
    """Owns one gva_ctx (bound to the device current at creation)."""

    def __init__(self, H, G, d_v, d_n, d_r, cache_dtype, rope_base=10000.0, scale=0.0):
        code = {"f32": GVA_F32, torch.float32: GVA_F32, "bf16": GVA_BF16, torch.bfloat16: GVA_BF16,
                "fp8": GVA_FP8_E4M3}[cache_dtype]
        self.dims = gva_dims(H, G, d_v, d_n, d_r, BLOCK_TOKENS, code, rope_base, scale)
        self.fp8 = code == GVA_FP8_E4M3
        # dtype of the new values and keys, and of the positional-key pool (bf16 for the fp8 cache)
        self.cache_torch_dtype = torch.float32 if code == GVA_F32 else torch.bfloat16
        # dtype of the value pool: the fp8 cache's is bytes (E4M3 codes, then int8 exponents)
        self.v_pool_dtype = torch.uint8 if self.fp8 else self.cache_torch_dtype
        h = C.c_void_p()
        _check(load().gva_create(C.byref(self.dims), C.byref(h)), "gva_create")
        self.handle = h

    def close(self):
        if self.handle:
            load().gva_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def H(self):
        return self.dims.H


def gva_create(H, G, d_v, d_n, d_r, cache_dtype="bf16", rope_base=10000.0, scale=0.0):
    return Context(H, G, d_v, d_n, d_r, cache_dtype, rope_base, scale)


def gva_destroy(ctx):
    ctx.close()


def _shape(t, shape, name):
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def fp8_value_pool_bytes(num_blocks, G, d_v):
    """Bytes of an fp8 value pool of num_blocks blocks: the E4M3 codes [NB][G][64][d_v], then the
    int8 scale exponents [NB][G][64]."""
    return num_blocks * G * BLOCK_TOKENS * (d_v + 1)


def fp8_pool_views(v_pool, G, d_v):
    """(codes [NB,G,64,d_v] uint8, exponents [NB,G,64] int8): views of an fp8 value pool."""
    NB = v_pool.numel() // (G * BLOCK_TOKENS * (d_v + 1))
    flat = v_pool.reshape(-1)
    n = NB * G * BLOCK_TOKENS * d_v
    return flat[:n].view(NB, G, BLOCK_TOKENS, d_v), flat[n:n + NB * G * BLOCK_TOKENS].view(torch.int8).view(
        NB, G, BLOCK_TOKENS)


def _num_blocks(ctx, v_pool):
    d = ctx.dims
    if ctx.fp8:
        per = d.G * BLOCK_TOKENS * (d.d_v + 1)
        if v_pool.numel() % per:
            raise ValueError(f"fp8 value pool of {v_pool.numel()} bytes is not a whole number of {per}-byte blocks")
        return v_pool.numel() // per
    return v_pool.shape[0]


def _check_pools(ctx, v_pool, kr_pool, k_pool=None):
    d = ctx.dims
    NB = _num_blocks(ctx, v_pool)
    if not ctx.fp8:
        _shape(v_pool, (NB, d.G, BLOCK_TOKENS, d.d_v), "v_pool")
    if k_pool is not None:
        _shape(k_pool, (NB, d.G, BLOCK_TOKENS, d.d_v), "k_pool")
    if d.d_r > 0 and kr_pool is not None:
        _shape(kr_pool, (NB, BLOCK_TOKENS, d.d_r), "kr_pool")
    return NB


def _check_table(block_table, B, seq_lens=None):
    if block_table.dim() != 2 or block_table.shape[0] < B:
        raise ValueError("block_table must be [>=B, max_blocks]")
    if seq_lens is not None and (seq_lens.dim() != 1 or seq_lens.shape[0] < B):
        raise ValueError("seq_lens must be [>=B]")


def gva_absorb_query(ctx, q_c, q_r, pos_q, M, q_abs, q_rot, stream=None):
    B = q_c.shape[0]
    d = ctx.dims
    _shape(q_c, (B, d.H, d.d_n), "q_c")
    _shape(M, (d.H, d.d_v, d.d_n), "M")
    _shape(q_abs, (B, d.H, d.d_v), "q_abs")
    _shape(pos_q, (B,), "pos_q")
    has_r = d.d_r > 0
    if has_r:
        _shape(q_r, (B, d.H, d.d_r), "q_r")
        _shape(q_rot, (B, d.H, d.d_r), "q_rot")
    _check(load().gva_absorb_query(ctx.handle, B, _ptr(q_c, torch.float32, "q_c"),
                                   _ptr(q_r, torch.float32, "q_r", allow_none=not has_r),
                                   _ptr(pos_q, torch.int32, "pos_q"), _ptr(M, torch.float32, "M"),
                                   _ptr(q_abs, torch.float32, "q_abs"),
                                   _ptr(q_rot, torch.float32, "q_rot", allow_none=not has_r), _stream(stream)),
           "gva_absorb_query")


def gva_cache_append(ctx, v_new, kr_new, pos, block_table, v_pool, kr_pool, stream=None):
    d = ctx.dims
    B, n = v_new.shape[0], v_new.shape[1]
    _shape(v_new, (B, n, d.G, d.d_v), "v_new")
    _shape(pos, (B,), "pos")
    _check_table(block_table, B)
    dt = ctx.cache_torch_dtype
    has_r = d.d_r > 0
    if has_r:
        _shape(kr_new, (B, n, d.d_r), "kr_new")
    _check_pools(ctx, v_pool, kr_pool if has_r else None)
    _check(load().gva_cache_append(ctx.handle, B, n, _ptr(v_new, dt, "v_new"),
                                   _ptr(kr_new, dt, "kr_new", allow_none=not has_r), _ptr(pos, torch.int32, "pos"),
                                   _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                   _num_blocks(ctx, v_pool), _ptr(v_pool, ctx.v_pool_dtype, "v_pool"),
                                   _ptr(kr_pool, dt, "kr_pool", allow_none=not has_r), _stream(stream)),
           "gva_cache_append")


def gva_decode_workspace_size(ctx, B, max_seq_len):
    return int(load().gva_decode_workspace_size(ctx.handle, int(B), int(max_seq_len)))


def gva_decode_attention(ctx, q_abs, q_rot, v_pool, kr_pool, block_table, seq_lens, max_seq_len, out, workspace,
                         stream=None):
    d = ctx.dims
    B = q_abs.shape[0]
    dt = ctx.cache_torch_dtype
    has_r = d.d_r > 0
    _shape(q_abs, (B, d.H, d.d_v), "q_abs")
    _shape(out, (B, d.H, d.d_v), "out")
    if has_r:
        _shape(q_rot, (B, d.H, d.d_r), "q_rot")
    _check_table(block_table, B, seq_lens)
    _check_pools(ctx, v_pool, kr_pool if has_r else None)
    _check(load().gva_decode_attention(ctx.handle, B, _ptr(q_abs, torch.float32, "q_abs"),
                                       _ptr(q_rot, torch.float32, "q_rot", allow_none=not has_r),
                                       _ptr(v_pool, ctx.v_pool_dtype, "v_pool"), _ptr(kr_pool, dt, "kr_pool", allow_none=not has_r),
                                       _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                       _num_blocks(ctx, v_pool), _ptr(seq_lens, torch.int32, "seq_lens"), int(max_seq_len),
                                       _ptr(out, torch.float32, "out"), _ptr(workspace, None, "workspace"),
                                       workspace.numel() * workspace.element_size(), _stream(stream)),
           "gva_decode_attention")


def gva_decode_partial(ctx, q_abs, q_rot, v_pool, kr_pool, block_table, seq_lens, max_seq_len, workspace,
                       stream=None):
    """The split-T pass of gva_decode_attention alone; its results stay in the workspace."""
    d = ctx.dims
    B = q_abs.shape[0]
    dt = ctx.cache_torch_dtype
    has_r = d.d_r > 0
    _shape(q_abs, (B, d.H, d.d_v), "q_abs")
    if has_r:
        _shape(q_rot, (B, d.H, d.d_r), "q_rot")
    _check_table(block_table, B, seq_lens)
    _check_pools(ctx, v_pool, kr_pool if has_r else None)
    _check(load().gva_decode_partial(ctx.handle, B, _ptr(q_abs, torch.float32, "q_abs"),
                                     _ptr(q_rot, torch.float32, "q_rot", allow_none=not has_r),
                                     _ptr(v_pool, ctx.v_pool_dtype, "v_pool"), _ptr(kr_pool, dt, "kr_pool", allow_none=not has_r),
                                     _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                     _num_blocks(ctx, v_pool), _ptr(seq_lens, torch.int32, "seq_lens"), int(max_seq_len),
                                     _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
                                     _stream(stream)),
           "gva_decode_partial")


def gva_decode_combine(ctx, B, max_seq_len, out, workspace, stream=None):
    """The combine pass: merges the partial results of the preceding gva_decode_partial into out."""
    d = ctx.dims
    _shape(out, (B, d.H, d.d_v), "out")
    _check(load().gva_decode_combine(ctx.handle, int(B), int(max_seq_len), _ptr(out, torch.float32, "out"),
                                     _ptr(workspace, None, "workspace"),
                                     workspace.numel() * workspace.element_size(), _stream(stream)),
           "gva_decode_combine")


def gva_decode_workspace_size_multi(ctx, B, n_q, max_seq_len):
    return int(load().gva_decode_workspace_size_multi(ctx.handle, int(B), int(n_q), int(max_seq_len)))


def gva_decode_attention_multi(ctx, q_abs, q_rot, v_pool, kr_pool, block_table, seq_lens, max_seq_len, out, workspace,
                               stream=None):
    """n_q query tokens per sequence (the last n_q positions), q_abs [B,n_q,H,d_v]; query i reads
    positions 0..seq_lens[b]-n_q+i.  out [B,n_q,H,d_v]."""
    d = ctx.dims
    B, n_q = q_abs.shape[0], q_abs.shape[1]
    dt = ctx.cache_torch_dtype
    has_r = d.d_r > 0
    _shape(q_abs, (B, n_q, d.H, d.d_v), "q_abs")
    _shape(out, (B, n_q, d.H, d.d_v), "out")
    if has_r:
        _shape(q_rot, (B, n_q, d.H, d.d_r), "q_rot")
    _check_table(block_table, B, seq_lens)
    _check_pools(ctx, v_pool, kr_pool if has_r else None)
    _check(load().gva_decode_attention_multi(ctx.handle, B, n_q, _ptr(q_abs, torch.float32, "q_abs"),
                                             _ptr(q_rot, torch.float32, "q_rot", allow_none=not has_r),
                                             _ptr(v_pool, ctx.v_pool_dtype, "v_pool"),
                                             _ptr(kr_pool, dt, "kr_pool", allow_none=not has_r),
                                             _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                             _num_blocks(ctx, v_pool), _ptr(seq_lens, torch.int32, "seq_lens"),
                                             int(max_seq_len), _ptr(out, torch.float32, "out"),
                                             _ptr(workspace, None, "workspace"),
                                             workspace.numel() * workspace.element_size(), _stream(stream)),
           "gva_decode_attention_multi")


def gva_decode_attention_noalloc(ctx, q_abs, q_rot, v_pool, kr_pool, block_table, seq_lens, max_seq_len, out,
                                 stream=None):
    """gva_decode_attention without a workspace, for callers that cannot allocate device memory:
    the library's fixed per-device scratch (NOALLOC_SCRATCH_BYTES) is used instead.  Calls on one
    device share it, so calls that may overlap on the GPU race; oversized batches raise
    GVAError with GVA_ERR_WORKSPACE."""
    d = ctx.dims
    B = q_abs.shape[0]
    dt = ctx.cache_torch_dtype
    has_r = d.d_r > 0
    _shape(q_abs, (B, d.H, d.d_v), "q_abs")
    _shape(out, (B, d.H, d.d_v), "out")
    if has_r:
        _shape(q_rot, (B, d.H, d.d_r), "q_rot")
    _check_table(block_table, B, seq_lens)
    _check_pools(ctx, v_pool, kr_pool if has_r else None)
    _check(load().gva_decode_attention_noalloc(ctx.handle, B, _ptr(q_abs, torch.float32, "q_abs"),
                                               _ptr(q_rot, torch.float32, "q_rot", allow_none=not has_r),
                                               _ptr(v_pool, ctx.v_pool_dtype, "v_pool"),
                                               _ptr(kr_pool, dt, "kr_pool", allow_none=not has_r),
                                               _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                               _num_blocks(ctx, v_pool), _ptr(seq_lens, torch.int32, "seq_lens"),
                                               int(max_seq_len), _ptr(out, torch.float32, "out"), _stream(stream)),
           "gva_decode_attention_noalloc")


def gva_decode_step_workspace_size(ctx, B, max_seq_len):
    return int(load().gva_decode_step_workspace_size(ctx.handle, int(B), int(max_seq_len)))


def gva_decode_step(ctx, q_c, q_r, M, v_new, kr_new, v_pool, kr_pool, block_table, seq_lens, max_seq_len, out,
                    workspace, stream=None):
    """One decode step: appends each sequence's new token (v_new [B,G,d_v], kr_new [B,d_r], cache
    dtype) at position seq_lens[b]-1, absorbs and rotates the query (q_c [B,H,d_n], q_r [B,H,d_r],
    M [H,d_v,d_n]) at that position, and attends over the context including the new token
    into out [B,H,d_v].  seq_lens already count the new token.  q_c, q_r, v_new, kr_new and out
    may be pinned host tensors: the kernels then read and write them across the bus directly."""
    d = ctx.dims
    B = q_c.shape[0]
    dt = ctx.cache_torch_dtype
    has_r = d.d_r > 0
    _shape(q_c, (B, d.H, d.d_n), "q_c")
    _shape(M, (d.H, d.d_v, d.d_n), "M")
    _shape(v_new, (B, d.G, d.d_v), "v_new")
    _shape(out, (B, d.H, d.d_v), "out")
    if has_r:
        _shape(q_r, (B, d.H, d.d_r), "q_r")
        _shape(kr_new, (B, d.d_r), "kr_new")
    _check_table(block_table, B, seq_lens)
    _check_pools(ctx, v_pool, kr_pool if has_r else None)
    _check(load().gva_decode_step(ctx.handle, B, _ptr(q_c, torch.float32, "q_c", allow_pinned=True),
                                  _ptr(q_r, torch.float32, "q_r", allow_none=not has_r, allow_pinned=True),
                                  _ptr(M, torch.float32, "M"),
                                  _ptr(v_new, dt, "v_new", allow_pinned=True),
                                  _ptr(kr_new, dt, "kr_new", allow_none=not has_r, allow_pinned=True),
                                  _ptr(v_pool, ctx.v_pool_dtype, "v_pool"), _ptr(kr_pool, dt, "kr_pool", allow_none=not has_r),
                                  _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                  _num_blocks(ctx, v_pool), _ptr(seq_lens, torch.int32, "seq_lens"), int(max_seq_len),
                                  _ptr(out, torch.float32, "out", allow_pinned=True),
                                  _ptr(workspace, None, "workspace"),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
           "gva_decode_step")


def gva_step_is_fused(ctx, B, max_seq_len):
    """1 if gva_decode_step runs the fused kernel for this batch shape, 0 if the separate kernels,
    -1 if neither applies."""
    return int(load().gva_step_is_fused(ctx.handle, int(B), int(max_seq_len)))


def gva_decode_step_partial(ctx, q_c, q_r, M, v_new, kr_new, v_pool, kr_pool, block_table, seq_lens, max_seq_len,
                            workspace, stream=None):
    """The fused step's split-T pass alone; gva_decode_combine completes it."""
    d = ctx.dims
    B = q_c.shape[0]
    dt = ctx.cache_torch_dtype
    has_r = d.d_r > 0
    _shape(q_c, (B, d.H, d.d_n), "q_c")
    _shape(M, (d.H, d.d_v, d.d_n), "M")
    _shape(v_new, (B, d.G, d.d_v), "v_new")
    if has_r:
        _shape(q_r, (B, d.H, d.d_r), "q_r")
        _shape(kr_new, (B, d.d_r), "kr_new")
    _check_table(block_table, B, seq_lens)
    _check_pools(ctx, v_pool, kr_pool if has_r else None)
    _check(load().gva_decode_step_partial(ctx.handle, B, _ptr(q_c, torch.float32, "q_c"),
                                          _ptr(q_r, torch.float32, "q_r", allow_none=not has_r),
                                          _ptr(M, torch.float32, "M"), _ptr(v_new, dt, "v_new"),
                                          _ptr(kr_new, dt, "kr_new", allow_none=not has_r),
                                          _ptr(v_pool, ctx.v_pool_dtype, "v_pool"), _ptr(kr_pool, dt, "kr_pool", allow_none=not has_r),
                                          _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                          _num_blocks(ctx, v_pool), _ptr(seq_lens, torch.int32, "seq_lens"), int(max_seq_len),
                                          _ptr(workspace, None, "workspace"),
                                          workspace.numel() * workspace.element_size(), _stream(stream)),
           "gva_decode_step_partial")


def gva_decode_step_workspace_size_multi(ctx, B, n_q, max_seq_len):
    return int(load().gva_decode_step_workspace_size_multi(ctx.handle, int(B), int(n_q), int(max_seq_len)))


def gva_decode_step_multi(ctx, q_c, q_r, M, v_new, kr_new, v_pool, kr_pool, block_table, seq_lens, max_seq_len, out,
                          workspace, stream=None):
    """A decode step of n_q tokens per sequence: q_c [B,n_q,H,d_n], q_r [B,n_q,H,d_r],
    v_new [B,n_q,G,d_v], kr_new [B,n_q,d_r] (the last n_q positions, which seq_lens already
    count), out [B,n_q,H,d_v].  The step's inputs and out may be pinned host tensors."""
    d = ctx.dims
    B, n_q = q_c.shape[0], q_c.shape[1]
    dt = ctx.cache_torch_dtype
    has_r = d.d_r > 0
    _shape(q_c, (B, n_q, d.H, d.d_n), "q_c")
    _shape(M, (d.H, d.d_v, d.d_n), "M")
    _shape(v_new, (B, n_q, d.G, d.d_v), "v_new")
    _shape(out, (B, n_q, d.H, d.d_v), "out")
    if has_r:
        _shape(q_r, (B, n_q, d.H, d.d_r), "q_r")
        _shape(kr_new, (B, n_q, d.d_r), "kr_new")
    _check_table(block_table, B, seq_lens)
    _check_pools(ctx, v_pool, kr_pool if has_r else None)
    _check(load().gva_decode_step_multi(ctx.handle, B, n_q, _ptr(q_c, torch.float32, "q_c", allow_pinned=True),
                                        _ptr(q_r, torch.float32, "q_r", allow_none=not has_r, allow_pinned=True),
                                        _ptr(M, torch.float32, "M"), _ptr(v_new, dt, "v_new", allow_pinned=True),
                                        _ptr(kr_new, dt, "kr_new", allow_none=not has_r, allow_pinned=True),
                                        _ptr(v_pool, ctx.v_pool_dtype, "v_pool"),
                                        _ptr(kr_pool, dt, "kr_pool", allow_none=not has_r),
                                        _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                        _num_blocks(ctx, v_pool), _ptr(seq_lens, torch.int32, "seq_lens"), int(max_seq_len),
                                        _ptr(out, torch.float32, "out", allow_pinned=True),
                                        _ptr(workspace, None, "workspace"),
                                        workspace.numel() * workspace.element_size(), _stream(stream)),
           "gva_decode_step_multi")


def gva_set_step_mode(ctx, mode):
    _check(load().gva_set_step_mode(ctx.handle, int(mode)), "gva_set_step_mode")


def gqa_decode_attention(ctx, q, k_pool, v_pool, block_table, seq_lens, max_seq_len, out, workspace, stream=None):
    d = ctx.dims
    B = q.shape[0]
    dt = ctx.cache_torch_dtype
    _shape(q, (B, d.H, d.d_v), "q")
    _shape(out, (B, d.H, d.d_v), "out")
    _check_table(block_table, B, seq_lens)
    _check_pools(ctx, v_pool, None, k_pool)
    _check(load().gqa_decode_attention(ctx.handle, B, _ptr(q, torch.float32, "q"), _ptr(k_pool, dt, "k_pool"),
                                       _ptr(v_pool, ctx.v_pool_dtype, "v_pool"), _ptr(block_table, torch.int32, "block_table"),
                                       block_table.shape[1], _num_blocks(ctx, v_pool), _ptr(seq_lens, torch.int32, "seq_lens"),
                                       int(max_seq_len), _ptr(out, torch.float32, "out"),
                                       _ptr(workspace, None, "workspace"),
                                       workspace.numel() * workspace.element_size(), _stream(stream)),
           "gqa_decode_attention")


def gva_set_split_tokens(ctx, split_tokens):
    _check(load().gva_set_split_tokens(ctx.handle, int(split_tokens)), "gva_set_split_tokens")


def gva_set_decode_path(ctx, path):
    _check(load().gva_set_decode_path(ctx.handle, int(path)), "gva_set_decode_path")


def gva_decode_plan(ctx, B, max_seq_len):
    st, ms = C.c_int(), C.c_int()
    _check(load().gva_decode_plan(ctx.handle, int(B), int(max_seq_len), C.byref(st), C.byref(ms)), "gva_decode_plan")
    return st.value, ms.value


def gva_get_device_error(ctx):
    """Returns the device error bits (0 when clean) and clears them; synchronises the device."""
    bits = C.c_uint()
    st = load().gva_get_device_error(ctx.handle, C.byref(bits))
    if st not in (GVA_OK, GVA_ERR_DEVICE_INDEX):
        raise GVAError(st, "gva_get_device_error")
    return bits.value


def gva_version():
    return int(load().gva_version())
