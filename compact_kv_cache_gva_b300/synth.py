"""Seeded synthetic inputs for the GVA decode path.

This module holds no attention arithmetic: it only draws random numbers, casts them to the
cache dtype (round to nearest even, by torch) and builds block tables.  Tests, the smoke
check and the benchmark all take their inputs from here, so the CUDA path and the CPU
oracle always see identical values.

Workloads (the pages train a 350M model on FineWeb-Edu; no weights or data are used here,
these draws stand in for its activations):

  id  name               dtype B    H  G  d_v=d_n d_r T
  1   tiny-fp32          f32   1    4  2  32      16  256
  2   layer-350m-bf16    bf16  32   16 4  64      16  4096
  3   dr24-bf16          bf16  64   16 4  64      24  8192
  4   long-context-bf16  bf16  8    16 4  64      16  131072
  5   ragged-paged-bf16  bf16  128  32 8  128     24  U[512, 32768] (seed 1), shuffled table

Distributions: V, q_c, q_r and the raw positional key ~ N(0,1); M_h ~ N(0, 1/d_v)
(variance 1/d_v).  Draw order from one generator seeded with `seed`: V, k_r, q_c, q_r, M.
Ragged lengths come from a second generator seeded with 1 (randint(512, 32769)), and the
block shuffle is the next draw (randperm) from that same generator.
"""
import dataclasses
from dataclasses import dataclass, field
import math

import torch

BLOCK = 64


@dataclass(frozen=True)
class Workload:
    id: int
    name: str
    dtype: str  # "f32" | "bf16" | "fp8" (E4M3 value cache, bf16 positional keys)
    B: int
    H: int
    G: int
    d_v: int
    d_n: int
    d_r: int
    T: int = 0  # uniform length (0 when ragged)
    T_range: tuple = ()  # (lo, hi) inclusive for ragged lengths
    shuffled: bool = False
    rope_base: float = 10000.0

    @property
    def torch_dtype(self):
        """dtype of new values and keys, and of the positional-key pool (bf16 for the fp8 cache)."""
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self):
        return 4 if self.dtype == "f32" else 2

    @property
    def bytes_per_token(self):
        """Cache bytes of one token of one layer: values and positional key in the cache dtype;
        the fp8 cache holds G*d_v codes, G scale exponents and d_r bf16 key elements."""
        if self.dtype == "fp8":
            return self.G * self.d_v + self.G + 2 * self.d_r
        return (self.G * self.d_v + self.d_r) * self.elem_bytes

    @property
    def r(self):
        return self.H // self.G

    @property
    def max_seq_len(self):
        return self.T if self.T else self.T_range[1]

    def describe(self):
        d = dict(workload=self.name, B=self.B, H=self.H, G=self.G, d_v=self.d_v, d_n=self.d_n, d_r=self.d_r,
                 cache_dtype=self.dtype, block_tokens=BLOCK)
        if self.T:
            d["T"] = self.T
        else:
            d["T_range"] = list(self.T_range)
            d["table"] = "shuffled" if self.shuffled else "identity"
        return d


WORKLOADS = {
    1: Workload(1, "tiny-fp32", "f32", B=1, H=4, G=2, d_v=32, d_n=32, d_r=16, T=256),
    2: Workload(2, "layer-350m-bf16", "bf16", B=32, H=16, G=4, d_v=64, d_n=64, d_r=16, T=4096),
    3: Workload(3, "dr24-bf16", "bf16", B=64, H=16, G=4, d_v=64, d_n=64, d_r=24, T=8192),
    4: Workload(4, "long-context-bf16", "bf16", B=8, H=16, G=4, d_v=64, d_n=64, d_r=16, T=131072),
    5: Workload(5, "ragged-paged-bf16", "bf16", B=128, H=32, G=8, d_v=128, d_n=128, d_r=24,
                T_range=(512, 32768), shuffled=True),
}


def with_cache(w: Workload, dtype: str):
    """The same workload over another cache dtype, named for it (e.g. long-context-fp8)."""
    name = w.name.replace(w.dtype, dtype) if w.dtype in w.name else f"{w.name}-{dtype}"
    return dataclasses.replace(w, dtype=dtype, name=name)


def custom(name="custom", dtype="bf16", B=2, H=4, G=2, d_v=64, d_n=None, d_r=16, T=0, T_range=(), shuffled=False):
    return Workload(0, name, dtype, B=B, H=H, G=G, d_v=d_v, d_n=d_v if d_n is None else d_n, d_r=d_r, T=T,
                    T_range=tuple(T_range), shuffled=shuffled)


def seq_lens(w: Workload, seed_lens: int = 1):
    """Per-sequence context lengths [B] int32 (CPU)."""
    if w.T:
        return torch.full((w.B,), w.T, dtype=torch.int32)
    g = torch.Generator().manual_seed(seed_lens)
    lo, hi = w.T_range
    return torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)


def block_table(w: Workload, lens, seed_lens: int = 1, spare_blocks: int = 0):
    """Block table [B, max_blocks] int32 and pool block count.

    Each sequence owns ceil(T_b/64) blocks; unused table entries are -1.  With an identity
    table, sequence b's blocks follow those of sequence b-1.  With a shuffled table the
    physical ids are a random permutation (the draw after the lengths, same generator)."""
    lens = torch.as_tensor(lens, dtype=torch.int64)
    nblk = (lens + BLOCK - 1) // BLOCK
    total = int(nblk.sum())
    max_blocks = max(1, int(math.ceil(w.max_seq_len / BLOCK)))
    if w.shuffled:
        g = torch.Generator().manual_seed(seed_lens)
        if not w.T:
            lo, hi = w.T_range
            torch.randint(lo, hi + 1, (w.B,), generator=g)  # replay the length draw
        ids = torch.randperm(total + spare_blocks, generator=g)[:total]
    else:
        ids = torch.arange(total)
    table = torch.full((w.B, max_blocks), -1, dtype=torch.int32)
    off = 0
    for b in range(w.B):
        n = int(nblk[b])
        table[b, :n] = ids[off:off + n].to(torch.int32)
        off += n
    return table, total + spare_blocks


@dataclass
class RawStep:
    """Raw inputs of one decode step (cache-dtype values where they enter the cache)."""
    q_c: torch.Tensor     # [B*n_q,H,d_n] f32
    q_r: torch.Tensor     # [B*n_q,H,d_r] f32 (unrotated)
    M: torch.Tensor       # [H,d_v,d_n] f32
    pos_q: torch.Tensor   # [B*n_q] int32
    v_new: torch.Tensor   # [B,n,G,d_v] cache dtype
    kr_new: torch.Tensor  # [B,n,d_r] cache dtype (unrotated)
    pos_new: torch.Tensor  # [B] int32, position of the first new token


def raw_inputs(w: Workload, lens, n_new, seed=0, device="cpu", pos_new=None, n_q=1):
    """Draws V (n_new tokens per sequence), the raw positional key, q_c, q_r and M, in that order.

    With n_q > 1 there are n_q query rows per sequence (row b*n_q + i at position T_b - n_q + i,
    the last n_q positions); n_q = 1 gives one row per sequence at T_b - 1."""
    g = torch.Generator(device=device).manual_seed(seed)
    B, H, G, dv, dn, dr = w.B, w.H, w.G, w.d_v, w.d_n, w.d_r
    v = torch.randn((B, n_new, G, dv), generator=g, device=device).to(w.torch_dtype)
    kr = torch.randn((B, n_new, dr), generator=g, device=device).to(w.torch_dtype)
    q_c = torch.randn((B * n_q, H, dn), generator=g, device=device)
    q_r = torch.randn((B * n_q, H, dr), generator=g, device=device)
    M = torch.randn((H, dv, dn), generator=g, device=device) * (1.0 / math.sqrt(dv))
    lens = torch.as_tensor(lens, dtype=torch.int32)
    pos_q = (lens[:, None] - n_q + torch.arange(n_q, dtype=torch.int32)[None]).reshape(-1).to(torch.int32).to(device)
    if pos_new is None:
        pos_new = (lens - n_new).clamp(min=0).to(torch.int32)
    return RawStep(q_c, q_r, M, pos_q, v, kr, torch.as_tensor(pos_new, dtype=torch.int32).to(device))


@dataclass
class DecodeInputs:
    """A filled cache plus absorbed/rotated queries, drawn directly (decode-only tests and bench).

    The pools are random cache-dtype arrays: a rotated N(0,1) positional key is again N(0,1),
    and q' = M_h q_c with M_h ~ N(0,1/d_v), q_c ~ N(0,1) has unit variance per element, so
    these draws have the distributions of the full path."""
    v_pool: torch.Tensor       # [NB,G,64,d_v]
    kr_pool: torch.Tensor      # [NB,64,d_r]
    block_table: torch.Tensor  # [B,max_blocks] int32
    seq_lens: torch.Tensor     # [B] int32
    q_abs: torch.Tensor        # [B,H,d_v] f32
    q_rot: torch.Tensor        # [B,H,d_r] f32
    num_blocks: int = 0
    extra: dict = field(default_factory=dict)


def decode_inputs(w: Workload, seed=0, device="cpu", lens=None, spare_blocks=0, k_pool=False):
    lens = seq_lens(w) if lens is None else torch.as_tensor(lens, dtype=torch.int32)
    table, nb = block_table(w, lens, spare_blocks=spare_blocks)
    g = torch.Generator(device=device).manual_seed(seed)
    if w.dtype == "fp8":
        v_pool = fp8_value_pool(w, nb, g, device)
    else:
        v_pool = torch.randn((nb, w.G, BLOCK, w.d_v), generator=g, device=device).to(w.torch_dtype)
    kr_pool = torch.randn((nb, BLOCK, w.d_r), generator=g, device=device).to(w.torch_dtype)
    q_abs = torch.randn((w.B, w.H, w.d_v), generator=g, device=device)
    q_rot = torch.randn((w.B, w.H, w.d_r), generator=g, device=device)
    extra = {}
    if k_pool:
        # matching GQA comparison: a key cache with the value cache's shape, and a plain query
        extra["k_pool"] = torch.randn((nb, w.G, BLOCK, w.d_v), generator=g, device=device).to(w.torch_dtype)
        extra["q"] = torch.randn((w.B, w.H, w.d_v), generator=g, device=device)
    return DecodeInputs(v_pool, kr_pool, table.to(device), lens.to(device), q_abs, q_rot, nb, extra)


def fp8_value_pool(w: Workload, nb, g, device):
    """A filled fp8 value pool: the E4M3 codes [nb][G][64][d_v] followed by the int8 exponents
    [nb][G][64].  Values are N(0,1) draws; each row's exponent is drawn from {-8, -7, -6} (the
    exponent a row of 64 or 128 such values needs is about -7) and the codes are torch's E4M3
    cast of the draws times 2^-e, clamped to the format's range."""
    x = torch.randn((nb, w.G, BLOCK, w.d_v), generator=g, device=device)
    e = torch.randint(-8, -5, (nb, w.G, BLOCK), generator=g, device=device)
    codes = (x * torch.exp2(-e.float())[..., None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return torch.cat([codes.reshape(-1), e.to(torch.int8).view(torch.uint8).reshape(-1)])


def pool_bits(t: torch.Tensor):
    """Host numpy view of a cache tensor as the oracle reads it (float32, or uint16 bf16 bits)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.uint8:  # fp8 value pool: codes, then exponents (flat)
        return t.reshape(-1).numpy()
    raise TypeError(t.dtype)
