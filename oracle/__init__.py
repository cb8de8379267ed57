"""Python face of the fp64 CPU oracle (gva_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the package smoke check and the
benchmark's CPU-baseline leg, never by the library.  Arrays are numpy; pools are raw
cache-dtype arrays (float32, uint16 holding bf16 bit patterns, or for the fp8 cache's value
pool uint8: the E4M3 codes followed by the int8 exponents), exactly the bytes a cache would
hold.  Every call checks shapes and raises on a non-zero oracle status.
"""
import ctypes as C
import os

import numpy as np

from .build import build as _build

F32, BF16, FP8 = 0, 1, 2
BLOCK = 64

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build()
        L = C.CDLL(path)
        dp, ip, vp = C.POINTER(C.c_double), C.POINTER(C.c_int32), C.c_void_p
        L.oracle_e4m3_to_double.restype = C.c_double
        L.oracle_e4m3_to_double.argtypes = [C.c_uint8]
        L.oracle_double_to_e4m3.restype = C.c_uint8
        L.oracle_double_to_e4m3.argtypes = [C.c_double]
        L.oracle_fp8_exponent.restype = C.c_int
        L.oracle_fp8_exponent.argtypes = [C.c_double]
        L.oracle_fp8_exp_offset.restype = C.c_int64
        L.oracle_fp8_exp_offset.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int64, C.c_int, C.c_int]
        L.oracle_cache_bytes_per_token.restype = C.c_double
        L.oracle_cache_bytes_per_token.argtypes = [C.c_int] * 4
        L.oracle_bf16_to_double.restype = C.c_double
        L.oracle_bf16_to_double.argtypes = [C.c_uint16]
        L.oracle_double_to_bf16.restype = C.c_uint16
        L.oracle_double_to_bf16.argtypes = [C.c_double]
        L.oracle_rope.restype = None
        L.oracle_rope.argtypes = [dp, C.c_int, C.c_double, C.c_double, dp]
        L.oracle_absorb.argtypes = [C.c_int] * 5 + [C.c_double, dp, dp, ip, dp, dp, dp]
        L.oracle_v_offset.restype = C.c_int64
        L.oracle_v_offset.argtypes = [C.c_int, C.c_int, C.c_int64, C.c_int, C.c_int, C.c_int]
        L.oracle_kr_offset.restype = C.c_int64
        L.oracle_kr_offset.argtypes = [C.c_int, C.c_int64, C.c_int, C.c_int]
        L.oracle_append.argtypes = [C.c_int] * 6 + [C.c_double, vp, vp, ip, ip, C.c_int, C.c_int, vp, vp]
        L.oracle_cache_ratio.restype = C.c_double
        L.oracle_cache_ratio.argtypes = [C.c_int] * 3
        L.oracle_decode_one.argtypes = ([C.c_int] * 6 + [C.c_double, vp, vp, ip, C.c_int, C.c_int, ip,
                                        C.c_int, C.c_int, dp, dp, dp])
        L.oracle_decode.argtypes = ([C.c_int] * 7 + [C.c_double, vp, vp, ip, C.c_int, C.c_int, ip, dp, dp, dp])
        L.oracle_decode_multi.argtypes = ([C.c_int] * 8 + [C.c_double, vp, vp, ip, C.c_int, C.c_int, ip, dp, dp, dp])
        L.oracle_decode_split.argtypes = ([C.c_int] * 6 + [C.c_double, vp, vp, ip, C.c_int, C.c_int, ip,
                                          C.c_int, C.c_int, dp, dp, C.c_int, dp])
        L.oracle_decode_unabsorbed.argtypes = ([C.c_int] * 7 + [C.c_double, C.c_double, vp, vp, ip, C.c_int,
                                               C.c_int, ip, dp, dp, ip, dp, dp])
        L.oracle_gqa_decode_one.argtypes = ([C.c_int] * 4 + [C.c_double, vp, vp, ip, C.c_int, C.c_int, ip,
                                            C.c_int, C.c_int, dp, dp])
        L.oracle_set_threads.restype = None
        L.oracle_set_threads.argtypes = [C.c_int]
        L.oracle_get_threads.restype = C.c_int
        L.oracle_get_threads.argtypes = []
        _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _check(st, what):
    if st != 0:
        raise OracleError(f"{what}: oracle status {st}")


def _d(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(C.POINTER(C.c_double))


def _i(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(C.POINTER(C.c_int32))


def _pool(a):
    if a.dtype == np.float32:
        code = F32
    elif a.dtype == np.uint16:
        code = BF16
    elif a.dtype == np.uint8:
        code = FP8  # value pool of the fp8 cache: E4M3 codes, then the int8 exponents
    else:
        raise TypeError("pool arrays are float32, uint16 (bf16 bits) or uint8 (fp8 value pool)")
    if not a.flags.c_contiguous:
        raise ValueError("pool must be contiguous")
    return code, C.c_void_p(a.ctypes.data)


def num_blocks_of(v_pool, G, d_v):
    """Blocks in a value pool: [NB][G][64][d_v] elements, or for the fp8 cache NB*G*64*d_v
    codes followed by NB*G*64 exponents."""
    per_block = G * BLOCK * d_v + (G * BLOCK if v_pool.dtype == np.uint8 else 0)
    return v_pool.size // per_block


def e4m3_to_double(code):
    return lib().oracle_e4m3_to_double(int(code))


def double_to_e4m3(x):
    return lib().oracle_double_to_e4m3(float(x))


def fp8_exponent(amax):
    return lib().oracle_fp8_exponent(float(amax))


def fp8_exp_offset(G, d_v, num_blocks, blk, g, o):
    return lib().oracle_fp8_exp_offset(G, d_v, num_blocks, blk, g, o)


def cache_bytes_per_token(dtype, G, d_v, d_r):
    return lib().oracle_cache_bytes_per_token({"f32": F32, "bf16": BF16, "fp8": FP8}.get(dtype, dtype), G, d_v, d_r)


def bf16_to_double(bits):
    return lib().oracle_bf16_to_double(int(bits))


def double_to_bf16(x):
    return lib().oracle_double_to_bf16(float(x))


def rope(x, pos, base=10000.0):
    x, px = _d(x)
    y = np.empty_like(x)
    lib().oracle_rope(px, x.shape[-1], float(pos), float(base), y.ctypes.data_as(C.POINTER(C.c_double)))
    return y


def absorb(q_c, q_r, pos_q, M, base=10000.0):
    """q_c [B,H,d_n], q_r [B,H,d_r], pos_q [B], M [H,d_v,d_n] -> (q_abs [B,H,d_v], q_rot [B,H,d_r])."""
    q_c, pqc = _d(q_c)
    q_r, pqr = _d(q_r)
    pos_q, pp = _i(pos_q)
    M, pM = _d(M)
    B, H, d_n = q_c.shape
    d_v = M.shape[1]
    d_r = q_r.shape[2]
    assert M.shape == (H, d_v, d_n) and q_r.shape[:2] == (B, H) and pos_q.shape == (B,)
    qa = np.empty((B, H, d_v))
    qo = np.empty((B, H, d_r))
    _check(lib().oracle_absorb(B, H, d_v, d_n, d_r, float(base), pqc, pqr, pp, pM,
                               qa.ctypes.data_as(C.POINTER(C.c_double)),
                               qo.ctypes.data_as(C.POINTER(C.c_double))), "absorb")
    return qa, qo


def v_offset(G, d_v, blk, g, o, i):
    return lib().oracle_v_offset(G, d_v, blk, g, o, i)


def kr_offset(d_r, blk, o, c):
    return lib().oracle_kr_offset(d_r, blk, o, c)


def append(v_new, kr_new, pos, block_table, v_pool, kr_pool, base=10000.0, raise_on_index=True):
    """In place on host pools.  v_new [B,n,G,d_v], kr_new [B,n,d_r] in the pool's dtype (for the
    fp8 cache, whose value pool is uint8, both are bf16 bits and the values are quantised).
    Returns the oracle status (0, or 5 when some slot could not be resolved)."""
    code, pv = _pool(v_pool)
    code2, pk = _pool(kr_pool)
    if code == FP8:
        assert code2 == BF16 and v_new.dtype == np.uint16 and kr_new.dtype == np.uint16
    else:
        assert code == code2 and v_new.dtype == v_pool.dtype and kr_new.dtype == kr_pool.dtype
    v_new = np.ascontiguousarray(v_new)
    kr_new = np.ascontiguousarray(kr_new)
    B, n, G, d_v = v_new.shape
    d_r = kr_new.shape[2]
    pos, ppos = _i(pos)
    bt, pbt = _i(block_table)
    max_blocks = bt.shape[1]
    num_blocks = num_blocks_of(v_pool, G, d_v)
    st = lib().oracle_append(code, B, n, G, d_v, d_r, float(base), C.c_void_p(v_new.ctypes.data),
                             C.c_void_p(kr_new.ctypes.data), ppos, pbt, max_blocks, num_blocks, pv, pk)
    if raise_on_index:
        _check(st, "append")
    return st


def cache_ratio(G, d_v, d_r):
    return lib().oracle_cache_ratio(G, d_v, d_r)


def _decode_common(v_pool, kr_pool, block_table, seq_lens, G, d_v):
    code, pv = _pool(v_pool)
    if kr_pool is None or kr_pool.size == 0:
        pk = C.c_void_p(v_pool.ctypes.data)  # never read when d_r == 0
    else:
        code2, pk = _pool(kr_pool)
        assert code2 == (BF16 if code == FP8 else code)
    bt, pbt = _i(block_table)
    sl, psl = _i(seq_lens)
    num_blocks = num_blocks_of(v_pool, G, d_v)
    return code, pv, pk, bt, pbt, sl, psl, num_blocks


def decode(q_abs, q_rot, v_pool, kr_pool, block_table, seq_lens, G, d_n=None, scale=0.0):
    """Full output [B,H,d_v] (fp64)."""
    q_abs, pqa = _d(q_abs)
    q_rot, pqr = _d(q_rot)
    B, H, d_v = q_abs.shape
    d_r = q_rot.shape[2]
    d_n = d_v if d_n is None else d_n
    code, pv, pk, bt, pbt, sl, psl, nb = _decode_common(v_pool, kr_pool, block_table, seq_lens, G, d_v)
    out = np.empty((B, H, d_v))
    _check(lib().oracle_decode(code, B, H, G, d_v, d_n, d_r, float(scale), pv, pk, pbt, bt.shape[1], nb, psl,
                               pqa, pqr, out.ctypes.data_as(C.POINTER(C.c_double))), "decode")
    return out


def decode_multi(q_abs, q_rot, v_pool, kr_pool, block_table, seq_lens, G, d_n=None, scale=0.0):
    """n_q queries per sequence, q_abs [B,n_q,H,d_v], q_rot [B,n_q,H,d_r]: query i of sequence b
    reads positions 0..seq_lens[b]-n_q+i.  Output [B,n_q,H,d_v] (fp64)."""
    q_abs, pqa = _d(q_abs)
    q_rot, pqr = _d(q_rot)
    B, n_q, H, d_v = q_abs.shape
    d_r = q_rot.shape[3]
    d_n = d_v if d_n is None else d_n
    code, pv, pk, bt, pbt, sl, psl, nb = _decode_common(v_pool, kr_pool, block_table, seq_lens, G, d_v)
    out = np.empty((B, n_q, H, d_v))
    _check(lib().oracle_decode_multi(code, B, n_q, H, G, d_v, d_n, d_r, float(scale), pv, pk, pbt, bt.shape[1], nb,
                                     psl, pqa, pqr, out.ctypes.data_as(C.POINTER(C.c_double))), "decode_multi")
    return out


def decode_one(q_abs, q_rot, v_pool, kr_pool, block_table, seq_lens, G, b, h, d_n=None, scale=0.0):
    """One output row (b, h), for sampling large workloads."""
    q_abs, pqa = _d(q_abs)
    q_rot, pqr = _d(q_rot)
    B, H, d_v = q_abs.shape
    d_r = q_rot.shape[2]
    d_n = d_v if d_n is None else d_n
    code, pv, pk, bt, pbt, sl, psl, nb = _decode_common(v_pool, kr_pool, block_table, seq_lens, G, d_v)
    out = np.empty(d_v)
    _check(lib().oracle_decode_one(code, H, G, d_v, d_n, d_r, float(scale), pv, pk, pbt, bt.shape[1], nb, psl,
                                   int(b), int(h), pqa, pqr, out.ctypes.data_as(C.POINTER(C.c_double))),
           "decode_one")
    return out


def decode_split(q_abs, q_rot, v_pool, kr_pool, block_table, seq_lens, G, b, h, S, d_n=None, scale=0.0):
    q_abs, pqa = _d(q_abs)
    q_rot, pqr = _d(q_rot)
    B, H, d_v = q_abs.shape
    d_r = q_rot.shape[2]
    d_n = d_v if d_n is None else d_n
    code, pv, pk, bt, pbt, sl, psl, nb = _decode_common(v_pool, kr_pool, block_table, seq_lens, G, d_v)
    out = np.empty(d_v)
    _check(lib().oracle_decode_split(code, H, G, d_v, d_n, d_r, float(scale), pv, pk, pbt, bt.shape[1], nb, psl,
                                     int(b), int(h), pqa, pqr, int(S), out.ctypes.data_as(C.POINTER(C.c_double))),
           "decode_split")
    return out


def decode_unabsorbed(q_c, q_r, pos_q, M, v_pool, kr_pool, block_table, seq_lens, G, scale=0.0, base=10000.0):
    q_c, pqc = _d(q_c)
    q_r, pqr = _d(q_r)
    pos_q, pp = _i(pos_q)
    M, pM = _d(M)
    B, H, d_n = q_c.shape
    d_v = M.shape[1]
    d_r = q_r.shape[2]
    code, pv, pk, bt, pbt, sl, psl, nb = _decode_common(v_pool, kr_pool, block_table, seq_lens, G, d_v)
    out = np.empty((B, H, d_v))
    _check(lib().oracle_decode_unabsorbed(code, B, H, G, d_v, d_n, d_r, float(scale), float(base), pv, pk, pbt,
                                          bt.shape[1], nb, psl, pqc, pqr, pp, pM,
                                          out.ctypes.data_as(C.POINTER(C.c_double))), "decode_unabsorbed")
    return out


def gqa_decode_one(q, k_pool, v_pool, block_table, seq_lens, G, b, h, scale=0.0):
    q, pq = _d(q)
    B, H, d = q.shape
    code, pv = _pool(v_pool)
    code2, pk = _pool(k_pool)
    assert code == code2
    bt, pbt = _i(block_table)
    sl, psl = _i(seq_lens)
    nb = v_pool.size // (G * BLOCK * d)
    out = np.empty(d)
    _check(lib().oracle_gqa_decode_one(code, H, G, d, float(scale), pk, pv, pbt, bt.shape[1], nb, psl, int(b),
                                       int(h), pq, out.ctypes.data_as(C.POINTER(C.c_double))), "gqa_decode_one")
    return out


def set_threads(n):
    lib().oracle_set_threads(int(n))


def get_threads():
    return lib().oracle_get_threads()
