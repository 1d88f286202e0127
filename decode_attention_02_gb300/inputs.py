"""Seeded synthetic inputs for MFA decode attention.

This module only draws and lays out data; it holds none of the attention
arithmetic.  The same generator feeds the CPU oracle (tests) and the CUDA path
(tests, benchmark, smoke run), so both sides see identical bytes.

Workload shapes follow the Step-3 MFA decode step (paperlayer.ai/abs/2507.19427v1,
section 5 "Model-System Co-design"): 64 query heads of width 256 attend over one
shared K head and one shared V head; the printed arithmetic intensity (128 with
8-bit KV) and effective rank (16,384) fix H=64 and d=256.  The KV cache is paged
with 64-token pages.

Recipe (fixed seeds, numpy PCG64 via ``default_rng``), in draw order:
  1. lengths: given, or uniform integers in [lo, hi] inclusive;
  2. physical page order: identity ("contiguous") or ``rng.permutation``;
  3. q ~ N(0,1) fp32 [B*T, H, d] (T new query tokens per sequence, 1 unless stated);
  4. K pool ~ N(0,1) fp32 [num_blocks, page, G*d] (G key/value heads per row, 1
     for MFA), drawn in chunks of ``_CHUNK_BLOCKS`` pages; optionally each
     scalar K element is multiplied by ``k_spike_mult`` with independent
     probability ``k_spike_frac`` (uniform draw right after each chunk's normals);
  5. V pool ~ N(0,1) fp32, same chunking, no spikes -- not drawn when one
     latent serves as keys and values (``kv_shared``): V is then the K pool.
Storage: bf16 by round-to-nearest-even, or FP8 e4m3 with one fp32 scale per
token row (absmax/448, 1 for an all-zero row), codes = e4m3(RNE(x/scale))
after clamping to +-448.  Unused page slots and unused physical pages are
filled with NaN when ``poison`` is set, so any read of them shows up.

KV append inputs (``append_step``): the case is drawn for the lengths after the step, and
each sequence's new bf16 key and value rows (``new_token_rows``, eight row kinds from N(0,1)
to all-zero, signed-zero, wide-range, huge and tiny rows) go to its last position.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

NUM_Q_HEADS = 64
HEAD_DIM = 256
PAGE_SIZE = 64
_CHUNK_BLOCKS = 512
BF16_NAN_BITS = 0x7FC0
E4M3_NAN_CODE = 0x7F


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    lens: Optional[Sequence[int]] = None        # explicit lengths, or None to draw
    len_range: Optional[tuple] = None           # (lo, hi) inclusive when drawn
    kv_dtype: str = "bf16"                      # "bf16" | "fp8_e4m3" | "mxfp4"
    layout: str = "shuffled"                    # "shuffled" | "contiguous"
    seed: int = 0
    k_spike_frac: float = 0.0
    k_spike_mult: float = 20.0
    extra_blocks: int = 0
    poison: bool = True
    num_q_heads: int = NUM_Q_HEADS
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    softmax_scale: Optional[float] = None       # None -> 1/sqrt(head_dim)
    tokens_per_seq: int = 1                     # T new query tokens per sequence (multi-token decode)
    num_kv_heads: int = 1                       # G key/value heads of width head_dim per cache row
    kv_shared: bool = False                     # True: one latent serves as keys and values

    def scale(self) -> float:
        if self.softmax_scale is not None:
            return float(self.softmax_scale)
        return 1.0 / math.sqrt(self.head_dim)


# The five decode workloads, plus the FP8 versions of the 4K and long shapes.
WORKLOADS = {
    "tiny_b1_l512_bf16": Workload(
        "tiny_b1_l512_bf16", batch=1, lens=(512,), layout="contiguous", seed=0),
    "b32_l4096_bf16": Workload(
        "b32_l4096_bf16", batch=32, lens=(4096,) * 32, seed=1),
    "ragged_b128_l1024_8192_bf16": Workload(
        "ragged_b128_l1024_8192_bf16", batch=128, len_range=(1024, 8192), seed=2,
        k_spike_frac=0.01, k_spike_mult=20.0),
    "b128_l4096_fp8": Workload(
        "b128_l4096_fp8", batch=128, lens=(4096,) * 128, kv_dtype="fp8_e4m3", seed=3),
    "long_b4_l131072_bf16": Workload(
        "long_b4_l131072_bf16", batch=4, lens=(131072, 131072, 65536, 16384), seed=4),
    "b32_l4096_fp8": Workload(
        "b32_l4096_fp8", batch=32, lens=(4096,) * 32, kv_dtype="fp8_e4m3", seed=5),
    "long_b4_l131072_fp8": Workload(
        "long_b4_l131072_fp8", batch=4, lens=(131072, 131072, 65536, 16384),
        kv_dtype="fp8_e4m3", seed=6),
    # multi-token decode: two new query tokens per sequence, causal among them
    "mtp2_b32_l4096_bf16": Workload(
        "mtp2_b32_l4096_bf16", batch=32, lens=(4096,) * 32, seed=7, tokens_per_seq=2),
    "mtp2_b32_l4096_fp8": Workload(
        "mtp2_b32_l4096_fp8", batch=32, lens=(4096,) * 32, kv_dtype="fp8_e4m3", seed=8, tokens_per_seq=2),
    # the attention designs the Step-3 page compares MFA with (section 5, "Attention Design";
    # section 7, attention ablation), at the 4K shape: grouped-query attention with 64 query
    # heads over 4 key/value heads of width 128 (effective rank 8,192), and a 512-wide latent
    # shared by keys and values under 128 query heads (intensity 512 with 8-bit KV)
    # 4-bit KV (MXFP4: E2M1 codes, one E8M0 scale per 32 elements of a row), the 4K shapes
    "b128_l4096_mxfp4": Workload(
        "b128_l4096_mxfp4", batch=128, lens=(4096,) * 128, kv_dtype="mxfp4", seed=11),
    "b32_l4096_mxfp4": Workload(
        "b32_l4096_mxfp4", batch=32, lens=(4096,) * 32, kv_dtype="mxfp4", seed=12),
    "gqa_b32_l4096_bf16": Workload(
        "gqa_b32_l4096_bf16", batch=32, lens=(4096,) * 32, seed=9, head_dim=128, num_kv_heads=4),
    "mla_b32_l4096_bf16": Workload(
        "mla_b32_l4096_bf16", batch=32, lens=(4096,) * 32, seed=10, num_q_heads=128, head_dim=512,
        kv_shared=True),
}


@dataclasses.dataclass
class Case:
    """Host tensors of one decode step (all torch CPU tensors, contiguous)."""
    workload: Workload
    q: torch.Tensor             # bf16 [B*T, H, d] (T = workload.tokens_per_seq)
    k_cache: torch.Tensor       # bf16 [nb, page, G*d] or uint8 e4m3 codes
    v_cache: torch.Tensor       # the same object as k_cache when the latent is shared
    k_scale: Optional[torch.Tensor]   # fp32 [nb, page] (FP8 only)
    v_scale: Optional[torch.Tensor]
    block_table: torch.Tensor   # int32 [B, max_pages], -1 where unused
    seq_lens: torch.Tensor      # int32 [B]

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def _pages(length: int, page: int) -> int:
    return (length + page - 1) // page


def _draw_pool(rng, nb, page, d, spike_frac, spike_mult):
    out = np.empty((nb, page, d), dtype=np.float32)
    for c0 in range(0, nb, _CHUNK_BLOCKS):
        c1 = min(nb, c0 + _CHUNK_BLOCKS)
        x = rng.standard_normal((c1 - c0, page, d), dtype=np.float32)
        if spike_frac > 0.0:
            mask = rng.random((c1 - c0, page, d), dtype=np.float32) < np.float32(spike_frac)
            x[mask] *= np.float32(spike_mult)
        out[c0:c1] = x
    return out


def _to_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x).to(torch.bfloat16)


# E2M1 magnitudes by code (OCP Microscaling FP4) and the midpoints between neighbours.
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_E2M1_MID = (_E2M1[1:] + _E2M1[:-1]) / 2


def _to_mxfp4(x: np.ndarray):
    """MXFP4 storage of rows of fp32 x [..., d]: codes uint8 [..., d/2] (element 2i in the low
    nibble of byte i) and E8M0 scales uint8 [..., d/32].  Per block of 32 elements the scale
    is 2^e, e = floor(log2(amax)) - 2 clamped to [-127, 127] (-127 for an all-zero block), and
    each element is rounded to the nearest E2M1 value of x / 2^e, ties to the even code,
    saturating at 6, sign kept."""
    *lead, d = x.shape
    blocks = x.reshape(*lead, d // 32, 32).astype(np.float32)
    amax = np.abs(blocks).max(axis=-1)
    _, E = np.frexp(amax)
    e = np.where(amax > 0, E - 3, -127).clip(-127, 127)
    y = np.ldexp(blocks.astype(np.float64), -e[..., None])
    a = np.abs(y)
    lo = np.searchsorted(_E2M1_MID, a, side="left")
    hi = np.searchsorted(_E2M1_MID, a, side="right")
    idx = np.minimum(np.where(lo != hi, lo + (lo % 2), lo), 7)
    code = (idx | np.where(np.signbit(y), 8, 0)).reshape(*lead, d).astype(np.uint8)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return torch.from_numpy(np.ascontiguousarray(packed)), torch.from_numpy((e + 127).astype(np.uint8))


def _to_e4m3(x: np.ndarray):
    """Per-token-row FP8 storage: codes (uint8) and fp32 scales absmax/448."""
    absmax = np.abs(x).max(axis=-1)
    scale = (absmax.astype(np.float32) / np.float32(448.0)).astype(np.float32)
    scale[absmax == 0] = np.float32(1.0)
    y = np.clip(x / scale[..., None], np.float32(-448.0), np.float32(448.0)).astype(np.float32)
    codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, torch.from_numpy(scale)


def generate(w: Workload, lens_override: Optional[Sequence[int]] = None) -> Case:
    """Draw one decode step's inputs for workload ``w`` (deterministic in w.seed)."""
    rng = np.random.default_rng(w.seed)
    B, H, d, page = w.batch, w.num_q_heads, w.head_dim, w.page_size
    if lens_override is not None:
        lens = np.asarray(lens_override, dtype=np.int64)
    elif w.lens is not None:
        lens = np.asarray(w.lens, dtype=np.int64)
    else:
        lo, hi = w.len_range
        lens = rng.integers(lo, hi + 1, size=B)
    assert lens.shape == (B,) and (lens >= 0).all()
    npages = [_pages(int(L), page) for L in lens]
    total = int(sum(npages))
    nb = max(1, total + w.extra_blocks)
    max_pages = max(1, max(npages) if npages else 1)

    if w.layout == "contiguous":
        perm = np.arange(nb, dtype=np.int64)
    else:
        perm = rng.permutation(nb)

    q = rng.standard_normal((B * w.tokens_per_seq, H, d), dtype=np.float32)
    row = w.num_kv_heads * d                    # cache row: G heads of width d side by side
    kf = _draw_pool(rng, nb, page, row, w.k_spike_frac, w.k_spike_mult)
    vf = kf if w.kv_shared else _draw_pool(rng, nb, page, row, 0.0, 1.0)

    table = np.full((B, max_pages), -1, dtype=np.int32)
    used = np.zeros(nb, dtype=bool)
    # (block, first unused slot) of each sequence's last page
    tails = []
    pos = 0
    for b in range(B):
        for p in range(npages[b]):
            blk = int(perm[pos]); pos += 1
            table[b, p] = blk
            used[blk] = True
        if npages[b]:
            rem = int(lens[b]) - page * (npages[b] - 1)
            if rem < page:
                tails.append((int(table[b, npages[b] - 1]), rem))

    if w.kv_dtype == "bf16":
        k_cache = _to_bf16(kf)
        v_cache = k_cache if w.kv_shared else _to_bf16(vf)
        k_scale = v_scale = None
        if w.poison:
            kb, vb = k_cache.view(torch.int16), v_cache.view(torch.int16)
            nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16)
            for blk, rem in tails:
                kb[blk, rem:] = nan
                vb[blk, rem:] = nan
            unused = torch.from_numpy(np.nonzero(~used)[0])
            if unused.numel():
                kb[unused] = nan
                vb[unused] = nan
    elif w.kv_dtype == "fp8_e4m3":
        k_cache, k_scale = _to_e4m3(kf)
        if w.kv_shared:
            v_cache, v_scale = k_cache, k_scale
        else:
            v_cache, v_scale = _to_e4m3(vf)
        if w.poison:
            for blk, rem in tails:
                k_cache[blk, rem:] = E4M3_NAN_CODE
                v_cache[blk, rem:] = E4M3_NAN_CODE
                k_scale[blk, rem:] = float("nan")
                v_scale[blk, rem:] = float("nan")
            unused = torch.from_numpy(np.nonzero(~used)[0])
            if unused.numel():
                k_cache[unused] = E4M3_NAN_CODE
                v_cache[unused] = E4M3_NAN_CODE
                k_scale[unused] = float("nan")
                v_scale[unused] = float("nan")
    elif w.kv_dtype == "mxfp4":
        k_cache, k_scale = _to_mxfp4(kf)
        if w.kv_shared:
            v_cache, v_scale = k_cache, k_scale
        else:
            v_cache, v_scale = _to_mxfp4(vf)
        if w.poison:
            # unused slots: code 6.0 everywhere and NaN scales (E8M0 255)
            for cache, sc in ((k_cache, k_scale), (v_cache, v_scale)):
                for blk, rem in tails:
                    cache[blk, rem:] = 0x77
                    sc[blk, rem:] = 255
                unused = torch.from_numpy(np.nonzero(~used)[0])
                if unused.numel():
                    cache[unused] = 0x77
                    sc[unused] = 255
    else:
        raise ValueError(f"unknown kv_dtype {w.kv_dtype!r}")

    return Case(
        workload=w,
        q=_to_bf16(q).contiguous(),
        k_cache=k_cache.contiguous(),
        v_cache=k_cache if w.kv_shared else v_cache.contiguous(),
        k_scale=None if k_scale is None else k_scale.contiguous(),
        v_scale=None if v_scale is None else v_scale.contiguous(),
        block_table=torch.from_numpy(table).contiguous(),
        seq_lens=torch.from_numpy(lens.astype(np.int32)).contiguous(),
    )


def small(name: str, batch: int, lens: Sequence[int], kv_dtype: str = "bf16", seed: int = 100,
          layout: str = "shuffled", extra_blocks: int = 2, k_spike_frac: float = 0.0,
          softmax_scale: Optional[float] = None, num_q_heads: int = NUM_Q_HEADS,
          head_dim: int = HEAD_DIM, page_size: int = PAGE_SIZE, tokens_per_seq: int = 1,
          num_kv_heads: int = 1, kv_shared: bool = False) -> Case:
    """A small poisoned case for parity tests (explicit lengths)."""
    w = Workload(name, batch=batch, lens=tuple(int(x) for x in lens), kv_dtype=kv_dtype,
                 layout=layout, seed=seed, extra_blocks=extra_blocks,
                 k_spike_frac=k_spike_frac, softmax_scale=softmax_scale,
                 num_q_heads=num_q_heads, head_dim=head_dim, page_size=page_size,
                 tokens_per_seq=tokens_per_seq, num_kv_heads=num_kv_heads, kv_shared=kv_shared)
    return generate(w)


# ------------------------------------------------------------------ new-token rows (KV append)

# Row kinds of new_token_rows, by row index modulo len(ROW_KINDS) (row 0 is "normal").
ROW_KINDS = ("normal", "zero", "signed_zero", "wide_range", "one_spike", "huge", "tiny", "spiky")


@dataclasses.dataclass
class AppendStep:
    """One decode step's new key/value rows and where they go."""
    k_new: torch.Tensor        # bf16 [B, d]
    v_new: torch.Tensor        # bf16 [B, d]
    positions: torch.Tensor    # int32 [B]: token index of the new row, -1 = no new token


def new_token_rows(batch: int, d: int = HEAD_DIM, seed: int = 0, kinds: Sequence[str] = ROW_KINDS) -> torch.Tensor:
    """Seeded bf16 [batch, d] rows covering the structures an FP8 row quantiser meets.

    Row r has kind kinds[r % len(kinds)], by default ROW_KINDS[r % 8]: N(0,1) ("normal"); all +0 ("zero"); a mix of +0
    and -0 ("signed_zero"); N(0,1) times 2^U[-20, 20] per element ("wide_range", many
    codes in the e4m3 subnormal range); N(0,1) * 1e-3 with one element 1e3 ("one_spike");
    N(0,1) * 1e30 ("huge"); N(0,1) * 1e-30 ("tiny"); N(0,1) with 1% of elements * 20
    ("spiky").  Values are drawn in fp32 and rounded to bf16 (nearest even).
    """
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((batch, d), dtype=np.float32)
    e = rng.integers(-20, 21, size=(batch, d))
    spike = rng.random((batch, d), dtype=np.float32) < np.float32(0.01)
    sign = rng.random((batch, d)) < 0.5
    where = rng.integers(0, d, size=batch)
    for r in range(batch):
        kind = kinds[r % len(kinds)]
        if kind == "zero":
            x[r] = 0.0
        elif kind == "signed_zero":
            x[r] = np.where(sign[r], np.float32(-0.0), np.float32(0.0))
        elif kind == "wide_range":
            x[r] = x[r] * np.exp2(e[r]).astype(np.float32)
        elif kind == "one_spike":
            x[r] *= np.float32(1e-3)
            x[r, where[r]] = np.float32(1e3)
        elif kind == "huge":
            x[r] *= np.float32(1e30)
        elif kind == "tiny":
            x[r] *= np.float32(1e-30)
        elif kind == "spiky":
            x[r, spike[r]] *= np.float32(20.0)
    return _to_bf16(x).contiguous()


def append_step(case: Case, seed: int = 0, inactive_every: int = 0,
                kinds: Sequence[str] = ROW_KINDS, tokens_per_seq: int = 1) -> AppendStep:
    """New rows for every sequence of ``case``, written at its last position(s).

    Build ``case`` for the lengths after the append (each sequence one token longer), so
    its block table already holds the page of the new token, as a serving system
    allocates it before the step; the slot's old contents are then overwritten.  With
    inactive_every = n > 0, every n-th sequence (b % n == n - 1) has no new token
    (position -1).  k rows use ``seed``, v rows ``seed + 1``; ``kinds`` as for
    new_token_rows (("normal",) for rows inside the FP8 decode's V-scale range).  With
    tokens_per_seq = T, each sequence gets T new rows ([B*T, d], sequence-major) at positions
    L - T .. L - 1; positions[b] is the first of them.
    """
    B = case.seq_lens.shape[0]
    d = case.q.shape[2]
    T = int(tokens_per_seq)
    pos = case.seq_lens.to(torch.int64) - T
    if inactive_every > 0:
        idx = torch.arange(B)
        pos[idx % inactive_every == inactive_every - 1] = -1
    pos[case.seq_lens < T] = -1
    return AppendStep(k_new=new_token_rows(B * T, d, seed, kinds), v_new=new_token_rows(B * T, d, seed + 1, kinds),
                      positions=pos.to(torch.int32).contiguous())
