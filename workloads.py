"""Seeded synthetic inputs for the KV hand-off: shapes, prompt lengths, block tables, values.

Both the CUDA path's tests/bench and the CPU oracle take their inputs from
here. This module holds no relayout arithmetic: it decides how big the pools
are, how long the prompts are, which physical blocks each side's allocator
hands out, and what bit patterns the prefill pool holds. It never computes a
slot, a shard or an address.

Block allocation follows pd.py on the page "PD 分离与 KV 传输" (section
"实现"): the prefill instance allocates ceil(n / Bp) blocks for a prompt of n
tokens and the decode instance reserves ceil((n + 1) / Bd), one slot more for
the first generated token. Physical block ids come from a seeded random
permutation of each pool, request after request, so a request's blocks are
scattered over the pool.

Pool layout (one buffer per TP shard): [L][C][N][B][H / T][D] elements of
``elem_bytes`` bytes, C = 2 for K and V, C = 1 for an MLA latent; a side with
more shards than KV heads (T > H, a multiple of H) holds one head per shard
([L][C][N][B][1][D]). Every shard's values are drawn independently, replicas
included.

The named workloads:

=========  ==============================================================
tiny       L2 C2 H2 D64 fp16 bit patterns; 1 x 100 tokens; 16 -> 32;
           TP1 -> TP1; 64 blocks per side                       (seed 0)
llama8b    L32 C2 H8 D128 bf16 N(0,1); 16 prompts U[512, 4096]; 16 -> 32;
           TP1 -> TP1; pools 1.25x the blocks needed             (seed 1)
llama70b   L80 C2 H8 D128 bf16 N(0,1); 1 x 4096; 16 -> 32; TP4 -> TP8;
           pools 1.25x                                           (seed 2)
qwen32k    L64 C2 H8 D128 bf16 N(0,1); 4 x 32768 (ragged variant:
           32768 - U[1, 63] each); 16 -> 64; TP4 -> TP2; 1.25x   (seed 3)
dsv3mla    L61 C1 H1 D576 bf16 N(0,1) latent; 64 prompts, lognormal
           (median 4096, sigma ln(4)/2), rounded, clipped to
           [1024, 16384]; 64 -> 16; TP1 -> TP1; 1.25x            (seed 4)
dsv3mla_   the same latent with TP8 on both sides, every shard holding
 tp8       the whole latent (read from the first prefill copy, written
           to all 8 decode copies); the first 8 prompts of the
           dsv3mla draw; 64 -> 16; 1.25x                         (seed 4)
=========  ==============================================================
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SENTINEL_BYTE = 0xFF          # decode pools start as all-ones bit patterns (0xFFFF for 16 bit)
POOL_SLACK = 1.25             # pools hold 1.25x the blocks the batch needs

_INT_DTYPES = {1: np.uint8, 2: np.uint16, 4: np.uint32}


def heads_per_shard(kv_heads: int, tp: int) -> int:
    """Head rows per token in one shard pool: H / T, or 1 when T > H."""
    return kv_heads // tp if tp <= kv_heads else 1


@dataclasses.dataclass(frozen=True, eq=False)
class Workload:
    name: str
    seed: int
    num_layers: int
    num_components: int
    kv_heads: int
    head_dim: int
    elem_bytes: int
    src_tp: int
    dst_tp: int
    src_block: int
    dst_block: int
    src_num_blocks: int
    dst_num_blocks: int
    seq_lens: np.ndarray          # int32 [R]
    src_off: np.ndarray           # int64 [R + 1], CSR into src_bt
    src_bt: np.ndarray            # int32, prefill block ids
    dst_off: np.ndarray           # int64 [R + 1], CSR into dst_bt
    dst_bt: np.ndarray            # int32, decode block ids
    values: str                   # "bits" (uniform bit patterns), "randn" (bf16 N(0,1)) or
                                  # "e4m3" (uniform over the 254 non-NaN E4M3 byte patterns)

    # -- shapes ---------------------------------------------------------
    @property
    def num_requests(self) -> int:
        return int(len(self.seq_lens))

    def src_shape(self):
        return (self.num_layers, self.num_components, self.src_num_blocks, self.src_block,
                heads_per_shard(self.kv_heads, self.src_tp), self.head_dim)

    def dst_shape(self):
        return (self.num_layers, self.num_components, self.dst_num_blocks, self.dst_block,
                heads_per_shard(self.kv_heads, self.dst_tp), self.head_dim)

    def src_pool_bytes(self) -> int:
        return int(np.prod(self.src_shape(), dtype=np.int64)) * self.elem_bytes

    def dst_pool_bytes(self) -> int:
        return int(np.prod(self.dst_shape(), dtype=np.int64)) * self.elem_bytes

    def int_dtype(self):
        return _INT_DTYPES[self.elem_bytes]

    def geometry(self) -> dict:
        """Keyword arguments shared by the oracle and the library binding."""
        return dict(num_layers=self.num_layers, num_components=self.num_components,
                    kv_heads=self.kv_heads, head_dim=self.head_dim,
                    elem_bytes=self.elem_bytes, src_tp=self.src_tp, dst_tp=self.dst_tp,
                    src_block=self.src_block, dst_block=self.dst_block,
                    src_num_blocks=self.src_num_blocks, dst_num_blocks=self.dst_num_blocks,
                    seq_lens=self.seq_lens, src_off=self.src_off, src_bt=self.src_bt,
                    dst_off=self.dst_off, dst_bt=self.dst_bt)

    def with_layers(self, num_layers: int) -> "Workload":
        """Same batch and tables with a different layer count (small profiling cases)."""
        return dataclasses.replace(self, name=f"{self.name}_L{num_layers}",
                                   num_layers=num_layers)

    # -- values ---------------------------------------------------------
    def src_pools_numpy(self):
        """Prefill pools on the host, one array per shard, filled from the seed."""
        rng = np.random.default_rng([self.seed, 1])
        out = []
        for _ in range(self.src_tp):
            if self.values == "randn":
                # bf16 = upper 16 bits of an fp32 N(0,1) sample (round to nearest even)
                f = rng.standard_normal(self.src_shape(), dtype=np.float32).view(np.uint32)
                rounded = f + 0x7FFF + ((f >> 16) & 1)
                out.append((rounded >> 16).astype(np.uint16))
            elif self.values == "e4m3":
                out.append(_finite_e4m3_codes(rng.integers(0, 254, size=self.src_shape(),
                                                            dtype=np.uint8)))
            else:
                info = np.iinfo(self.int_dtype())
                out.append(rng.integers(0, int(info.max) + 1, size=self.src_shape(),
                                        dtype=self.int_dtype()))
        return out

    def dst_pools_numpy(self, sentinel_byte: int = SENTINEL_BYTE):
        return [np.full(self.dst_shape(), self._sentinel_value(sentinel_byte),
                        dtype=self.int_dtype()) for _ in range(self.dst_tp)]

    def _sentinel_value(self, sentinel_byte: int) -> int:
        v = 0
        for _ in range(self.elem_bytes):
            v = (v << 8) | sentinel_byte
        return v

    def src_pools_torch(self, device):
        """Prefill pools on ``device`` (integer views of the element bits)."""
        import torch
        tdt = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[self.elem_bytes]
        g = torch.Generator(device=device)
        g.manual_seed(self.seed)
        out = []
        for _ in range(self.src_tp):
            if self.values == "randn":
                assert self.elem_bytes == 2
                t = torch.randn(self.src_shape(), generator=g, device=device,
                                dtype=torch.bfloat16)
                out.append(t.view(torch.int16))
            elif self.values == "e4m3":
                assert self.elem_bytes == 1
                r = torch.randint(0, 254, self.src_shape(), generator=g, device=device,
                                  dtype=torch.uint8)
                out.append(r + (r >= 0x7F).to(torch.uint8))
            else:
                lo, hi = {1: (0, 256), 2: (-32768, 32768), 4: (-2**31, 2**31)}[self.elem_bytes]
                out.append(torch.randint(lo, hi, self.src_shape(), generator=g, device=device,
                                         dtype=tdt))
        return out

    def dst_pools_torch(self, device, sentinel_byte: int = SENTINEL_BYTE):
        import torch
        out = []
        for _ in range(self.dst_tp):
            t = torch.empty(self.dst_pool_bytes(), dtype=torch.uint8, device=device)
            t.fill_(sentinel_byte)
            tdt = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[self.elem_bytes]
            out.append(t.view(tdt).view(self.dst_shape()))
        return out


def _finite_e4m3_codes(r):
    """Byte patterns 0..253 spread over the 254 bytes other than 0x7F and 0xFF (the
    two NaN patterns of an E4M3 element): r -> r, or r + 1 from 0x7F on."""
    return (r + (r >= 0x7F)).astype(np.uint8)


# -- block allocation -------------------------------------------------------

def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def allocate_tables(rng, seq_lens, block, num_blocks, reserve_extra: int, shared_prefix=0):
    """Seeded allocator: request after request takes the next ids of a permutation.

    Each request gets ceil((n + reserve_extra) / block) ids. With
    ``shared_prefix`` > 0, every request after the first reuses the first
    request's first ``shared_prefix`` ids (a cached common prefix: the same
    physical prefill blocks appear in several tables).
    """
    perm = rng.permutation(num_blocks).astype(np.int32)
    counts = [_ceil_div(int(n) + reserve_extra, block) if (n > 0 or reserve_extra) else 0
              for n in seq_lens]
    off = np.zeros(len(seq_lens) + 1, dtype=np.int64)
    tables, pos = [], 0
    for r, cnt in enumerate(counts):
        reuse = min(shared_prefix, cnt, len(tables[0]) if tables else 0) if r > 0 else 0
        fresh = cnt - reuse
        if pos + fresh > num_blocks:
            raise ValueError("pool too small for the batch")
        ids = np.concatenate([tables[0][:reuse], perm[pos:pos + fresh]]) if reuse else \
            perm[pos:pos + fresh]
        pos += fresh
        tables.append(ids.astype(np.int32))
        off[r + 1] = off[r] + cnt
    bt = np.concatenate(tables).astype(np.int32) if tables else np.zeros(0, np.int32)
    return off, bt


def blocks_needed(seq_lens, block, reserve_extra=0) -> int:
    return int(sum(_ceil_div(int(n) + reserve_extra, block) for n in seq_lens))


def custom(name, seed, *, num_layers, num_components, kv_heads, head_dim, elem_bytes,
           src_tp, dst_tp, src_block, dst_block, seq_lens, values="bits",
           src_num_blocks=None, dst_num_blocks=None, slack=POOL_SLACK, shared_prefix=0,
           dst_reserve=1) -> Workload:
    """Any geometry; lengths given; tables drawn from ``seed``."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(seq_lens, dtype=np.int32)
    need_s = blocks_needed(lens, src_block)
    need_d = blocks_needed(lens, dst_block, dst_reserve)
    np_ = src_num_blocks or max(1, math.ceil(slack * need_s))
    nd_ = dst_num_blocks or max(1, math.ceil(slack * need_d))
    s_off, s_bt = allocate_tables(rng, lens, src_block, np_, 0, shared_prefix)
    d_off, d_bt = allocate_tables(rng, lens, dst_block, nd_, dst_reserve)
    return Workload(name, seed, num_layers, num_components, kv_heads, head_dim, elem_bytes,
                    src_tp, dst_tp, src_block, dst_block, np_, nd_, lens, s_off, s_bt, d_off,
                    d_bt, values)


def tiny() -> Workload:
    rng = np.random.default_rng(0)
    lens = np.array([100], dtype=np.int32)
    s_off, s_bt = allocate_tables(rng, lens, 16, 64, 0)
    d_off, d_bt = allocate_tables(rng, lens, 32, 64, 1)
    return Workload("tiny", 0, 2, 2, 2, 64, 2, 1, 1, 16, 32, 64, 64, lens, s_off, s_bt,
                    d_off, d_bt, "bits")


def _named(name, seed, lens_fn, **geo) -> Workload:
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens_fn(rng), dtype=np.int32)
    need_s = blocks_needed(lens, geo["src_block"])
    need_d = blocks_needed(lens, geo["dst_block"], 1)
    np_ = math.ceil(POOL_SLACK * need_s)
    nd_ = math.ceil(POOL_SLACK * need_d)
    s_off, s_bt = allocate_tables(rng, lens, geo["src_block"], np_, 0)
    d_off, d_bt = allocate_tables(rng, lens, geo["dst_block"], nd_, 1)
    return Workload(name, seed, geo["num_layers"], geo["num_components"], geo["kv_heads"],
                    geo["head_dim"], 2, geo["src_tp"], geo["dst_tp"], geo["src_block"],
                    geo["dst_block"], np_, nd_, lens, s_off, s_bt, d_off, d_bt, "randn")


def llama8b() -> Workload:
    return _named("llama8b", 1, lambda rng: rng.integers(512, 4097, size=16),
                  num_layers=32, num_components=2, kv_heads=8, head_dim=128, src_tp=1,
                  dst_tp=1, src_block=16, dst_block=32)


def llama70b() -> Workload:
    return _named("llama70b", 2, lambda rng: [4096], num_layers=80, num_components=2,
                  kv_heads=8, head_dim=128, src_tp=4, dst_tp=8, src_block=16, dst_block=32)


def qwen32k(ragged: bool = False) -> Workload:
    def lens(rng):
        if ragged:
            return 32768 - rng.integers(1, 64, size=4)
        return [32768] * 4
    w = _named("qwen32k_ragged" if ragged else "qwen32k", 3, lens, num_layers=64,
               num_components=2, kv_heads=8, head_dim=128, src_tp=4, dst_tp=2, src_block=16,
               dst_block=64)
    return w


def dsv3mla() -> Workload:
    def lens(rng):
        x = rng.lognormal(mean=math.log(4096.0), sigma=math.log(4.0) / 2.0, size=64)
        return np.clip(np.rint(x), 1024, 16384).astype(np.int64)
    return _named("dsv3mla", 4, lens, num_layers=61, num_components=1, kv_heads=1,
                  head_dim=576, src_tp=1, dst_tp=1, src_block=64, dst_block=16)


def dsv3mla_tp8() -> Workload:
    """The MLA latent replicated over TP8 on both sides (8 prompts of the dsv3mla draw:
    8 decode copies of the whole batch stay within a few tens of GB)."""
    def lens(rng):
        x = rng.lognormal(mean=math.log(4096.0), sigma=math.log(4.0) / 2.0, size=64)
        return np.clip(np.rint(x), 1024, 16384).astype(np.int64)[:8]
    return _named("dsv3mla_tp8", 4, lens, num_layers=61, num_components=1, kv_heads=1,
                  head_dim=576, src_tp=8, dst_tp=8, src_block=64, dst_block=16)


NAMED = {
    "tiny": tiny,
    "llama8b": llama8b,
    "llama70b": llama70b,
    "qwen32k": qwen32k,
    "qwen32k_ragged": lambda: qwen32k(ragged=True),
    "dsv3mla": dsv3mla,
    "dsv3mla_tp8": dsv3mla_tp8,
}


def get(name: str) -> Workload:
    return NAMED[name]()
