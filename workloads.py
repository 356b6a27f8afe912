"""Seeded synthetic workloads for paged attention: the only module that both the
CUDA path's tests/bench and the CPU oracle take inputs from.

It draws shapes, contexts, page assignments and N(0,1) values; it holds none
of the attention arithmetic (no append, no softmax, no fp8 encoding: the fp8
scale below is the harness's calibration choice, handed unchanged to both
sides).  bf16 arrays are numpy ``uint16`` bit patterns, fp8 pools ``uint8``.

The shapes follow the workloads of the pages; the pages' own prompts and
evaluation queries are private, so these inputs stand in for their shapes only:
  tiny decode         4 sequences, contexts {5,33,64,100}, Hq 8 / Hkv 2, D 64, fp32, P 32, 16 pages
  batched decode      512 sequences, contexts U{64..2662}, Hq 16 / Hkv 8, D 128, bf16, P 32
  mixed step          256 decode rows (U{64..1024}) + a 256-row causal chunk at 1024 of a 2662-token prompt
  shared prefix       768 sequences, Hq 28 / Hkv 4, D 128, fp8 e4m3 K/V, bf16 Q, 128 + U{0..127} tokens,
                      70% sharing a 90-token prefix (its two full 32-token pages shared)
  long context        64 sequences x 32768 tokens, Hq 32 / Hkv 8, D 128, bf16, P 16, split-KV
  fp8 variants        the batched-decode and long-context shapes with e4m3 pools (per-tensor scales)
"""
from __future__ import annotations

import concurrent.futures as cf
import math
import os
from dataclasses import dataclass, field, replace

import numpy as np

F32, BF16, E4M3 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", BF16: "bf16", E4M3: "fp8_e4m3"}
ELT_SIZE = {F32: 4, BF16: 2, E4M3: 1}
POISON = {F32: 0x7FC00000, BF16: 0x7FC0, E4M3: 0x7F}  # quiet-NaN patterns for unwritten slots


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even) bit patterns, via torch's cast."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _cast(x: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == BF16:
        return to_bf16_bits(x)
    raise ValueError("inputs are drawn as f32 or bf16")


def as_f32(x: np.ndarray, dtype: int) -> np.ndarray:
    """Input array (f32 or bf16 bits) as float32 values."""
    return x.astype(np.float32) if dtype == F32 else bf16_bits_to_f32(x)


@dataclass
class Workload:
    name: str
    Hq: int
    Hkv: int
    D: int
    P: int
    kv_dtype: int
    in_dtype: int          # dtype of the appended k/v rows
    q_dtype: int
    num_pages: int
    block_tables: np.ndarray  # int32 [num_seqs][max_blocks], -1 = unused
    # history: rows appended before the step (setup, not timed)
    hist_seq: np.ndarray
    hist_pos: np.ndarray
    hist_k: np.ndarray
    hist_v: np.ndarray
    # the step: rows appended then attended
    seq_ids: np.ndarray
    positions: np.ndarray
    q: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    chunks: list = field(default_factory=list)  # [(row_begin, n_rows)]
    k_scale: float = 1.0
    v_scale: float = 1.0
    softmax_scale: float = 0.0
    shared_pages: int = 0   # physical pages referenced by more than one sequence
    description: str = ""

    @property
    def num_seqs(self) -> int:
        return int(self.block_tables.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def n_rows(self) -> int:
        return int(self.seq_ids.shape[0])

    @property
    def elt(self) -> int:
        return ELT_SIZE[self.kv_dtype]

    def decode_rows(self) -> np.ndarray:
        in_chunk = np.zeros(self.n_rows, dtype=bool)
        for b, n in self.chunks:
            in_chunk[b:b + n] = True
        return np.nonzero(~in_chunk)[0]

    # ---- algorithmic byte counts (valid token slots only, shared pages once) ----
    def kv_bytes_logical(self) -> int:
        """K+V bytes of every row's keys 0..position, counted per row and kv head."""
        L = self.positions.astype(np.int64) + 1
        return int(L.sum()) * self.Hkv * self.D * self.elt * 2

    def kv_bytes_unique(self) -> int:
        """K+V bytes of the distinct (page, slot) pairs the step reads.

        Rows of one sequence read nested key ranges, so each sequence counts
        once at its longest row; a physical page shared by several sequences
        counts once."""
        per_page = {}
        longest = {}
        for s, p in zip(self.seq_ids.tolist(), self.positions.tolist()):
            longest[s] = max(longest.get(s, -1), p + 1)
        for s, L in longest.items():
            for j in range((L + self.P - 1) // self.P):
                pg = int(self.block_tables[s, j])
                valid = min(self.P, L - j * self.P)
                per_page[pg] = max(per_page.get(pg, 0), valid)
        return sum(per_page.values()) * self.Hkv * self.D * self.elt * 2

    def qo_bytes(self) -> int:
        return 2 * self.n_rows * self.Hq * self.D * ELT_SIZE[self.q_dtype]

    def append_bytes(self) -> int:
        return self.n_rows * self.Hkv * self.D * 2 * (ELT_SIZE[self.in_dtype] + self.elt)

    def pool_shape(self):
        return (self.num_pages, self.Hkv, self.P, self.D)

    def empty_pool(self) -> np.ndarray:
        """A host pool with every slot poisoned with a quiet-NaN pattern."""
        np_t = {F32: np.uint32, BF16: np.uint16, E4M3: np.uint8}[self.kv_dtype]
        pool = np.full(self.pool_shape(), POISON[self.kv_dtype], dtype=np_t)
        if self.kv_dtype == F32:
            pool = pool.view(np.float32)
        return pool


# ----------------------------------------------------------------- helpers --

def _children(seed: int, n: int):
    return np.random.SeedSequence(seed).spawn(n)


def _normals(ss, shape) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    np.random.Generator(np.random.PCG64(ss)).standard_normal(out=out.reshape(-1), dtype=np.float32)
    return out


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _draw_rows(seed: int, counts, Hkv: int, D: int, dtype: int):
    """N(0,1) K and V rows for groups of rows, one child seed per group, in parallel."""
    total = int(sum(counts))
    np_t = np.float32 if dtype == F32 else np.uint16
    K = np.empty((total, Hkv, D), dtype=np_t)
    V = np.empty((total, Hkv, D), dtype=np_t)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    kids = _children(seed, len(counts))

    def fill(i):
        n = int(counts[i])
        if n == 0:
            return
        a, b = kids[i].spawn(2)
        K[offs[i]:offs[i] + n] = _cast(_normals(a, (n, Hkv, D)), dtype)
        V[offs[i]:offs[i] + n] = _cast(_normals(b, (n, Hkv, D)), dtype)

    with cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(len(counts))))
    return K, V


def _assign_pages(rng, pages_per_seq, num_pages, max_blocks):
    """Block tables from a shuffled pool: a random permutation of the physical
    pages handed out to the sequences in order; unused entries -1."""
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((len(pages_per_seq), max_blocks), -1, dtype=np.int32)
    k = 0
    for s, n in enumerate(pages_per_seq):
        bt[s, :n] = perm[k:k + n]
        k += n
    assert k <= num_pages
    return bt


def _decode_workload(name, seed, ctx, Hq, Hkv, D, P, kv_dtype, q_dtype, max_ctx, spare_pages,
                     description, num_pages=None):
    """Sequences with contexts ctx (keys attended, own token included): history
    rows 0..L-2 per sequence, then one decode row at position L-1."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.asarray(ctx, dtype=np.int64)
    n = len(ctx)
    max_blocks = (max_ctx + P - 1) // P
    pages = [int((L + P - 1) // P) for L in ctx]
    if num_pages is None:
        num_pages = sum(pages) + spare_pages
    bt = _assign_pages(rng, pages, num_pages, max_blocks)
    in_dtype = kv_dtype if kv_dtype != E4M3 else BF16
    hist_counts = [int(L - 1) for L in ctx]
    hist_seq = np.repeat(np.arange(n, dtype=np.int32), hist_counts)
    hist_pos = np.concatenate([np.arange(c, dtype=np.int32) for c in hist_counts]) if n else np.zeros(0, np.int32)
    hist_k, hist_v = _draw_rows(seed * 1000 + 1, hist_counts, Hkv, D, in_dtype)
    seq_ids = np.arange(n, dtype=np.int32)
    positions = (ctx - 1).astype(np.int32)
    q = _cast(rng.standard_normal((n, Hq, D), dtype=np.float32), q_dtype)
    k_new = _cast(rng.standard_normal((n, Hkv, D), dtype=np.float32), in_dtype)
    v_new = _cast(rng.standard_normal((n, Hkv, D), dtype=np.float32), in_dtype)
    return Workload(name=name, Hq=Hq, Hkv=Hkv, D=D, P=P, kv_dtype=kv_dtype, in_dtype=in_dtype,
                    q_dtype=q_dtype, num_pages=num_pages, block_tables=bt, hist_seq=hist_seq,
                    hist_pos=hist_pos, hist_k=hist_k, hist_v=hist_v, seq_ids=seq_ids,
                    positions=positions, q=q, k_new=k_new, v_new=v_new, description=description)


# ------------------------------------------------------------------ configs --

def tiny_decode(seed: int = 1) -> Workload:
    """4 sequences, contexts {5,33,64,100}, Hq 8 / Hkv 2, D 64, fp32, P 32, 16 pages."""
    return _decode_workload("tiny_decode", seed, [5, 33, 64, 100], 8, 2, 64, 32, F32, F32,
                            max_ctx=128, spare_pages=0, num_pages=16,
                            description="tiny decode: 4 seqs ctx {5,33,64,100}, Hq8/Hkv2, D64, fp32, P32, 16 pages")


def batched_decode(seed: int = 2, n_seqs: int = 512, ctx_lo: int = 64, ctx_hi: int = 2662) -> Workload:
    """n_seqs sequences with contexts U{ctx_lo..ctx_hi}, Hq 16 / Hkv 8, D 128, bf16, P 32."""
    rng = np.random.Generator(np.random.PCG64(seed + 100))
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=n_seqs)
    return _decode_workload("batched_decode", seed, ctx, 16, 8, 128, 32, BF16, BF16,
                            max_ctx=ctx_hi, spare_pages=64,
                            description=f"0.6B-class batched decode: {n_seqs} seqs ctx U[{ctx_lo},{ctx_hi}], "
                                        "Hq16/Hkv8, D128, bf16, P32, decode + append")


def long_context(seed: int = 5, n_seqs: int = 64, ctx: int = 32768) -> Workload:
    """n_seqs sequences of ctx tokens, Hq 32 / Hkv 8, D 128, bf16, P 16 (split-KV)."""
    return _decode_workload("long_context", seed, [ctx] * n_seqs, 32, 8, 128, 16, BF16, BF16,
                            max_ctx=ctx, spare_pages=0,
                            description=f"long-context split-KV: {n_seqs} seqs x {ctx} tokens, Hq32/Hkv8, "
                                        "D128, bf16, P16")


def _with_fp8_scales(wl: Workload) -> Workload:
    """Per-tensor fp8 scales: amax of every K (V) value the pools will hold, / 448, in fp32."""
    amax_k = max(np.abs(as_f32(wl.hist_k, wl.in_dtype)).max(initial=0.0), np.abs(as_f32(wl.k_new, wl.in_dtype)).max())
    amax_v = max(np.abs(as_f32(wl.hist_v, wl.in_dtype)).max(initial=0.0), np.abs(as_f32(wl.v_new, wl.in_dtype)).max())
    wl.k_scale = float(np.float32(amax_k) / np.float32(448.0))
    wl.v_scale = float(np.float32(amax_v) / np.float32(448.0))
    return wl


def batched_decode_fp8(seed: int = 2, n_seqs: int = 512, ctx_lo: int = 64, ctx_hi: int = 2662) -> Workload:
    """The batched-decode shape with an fp8 e4m3 K/V cache (bf16 rows in, per-tensor scales)."""
    rng = np.random.Generator(np.random.PCG64(seed + 100))
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=n_seqs)
    return _with_fp8_scales(_decode_workload(
        "batched_decode_fp8", seed, ctx, 16, 8, 128, 32, E4M3, BF16, max_ctx=ctx_hi, spare_pages=64,
        description=f"0.6B-class batched decode, fp8 K/V: {n_seqs} seqs ctx U[{ctx_lo},{ctx_hi}], Hq16/Hkv8, D128, "
                    "fp8 e4m3 K/V (per-tensor scale), bf16 Q, P32, decode + append"))


def long_context_fp8(seed: int = 5, n_seqs: int = 64, ctx: int = 32768) -> Workload:
    """The long-context shape with an fp8 e4m3 K/V cache (bf16 rows in, per-tensor scales)."""
    return _with_fp8_scales(_decode_workload(
        "long_context_fp8", seed, [ctx] * n_seqs, 32, 8, 128, 16, E4M3, BF16, max_ctx=ctx, spare_pages=0,
        description=f"long-context split-KV, fp8 K/V: {n_seqs} seqs x {ctx} tokens, Hq32/Hkv8, D128, "
                    "fp8 e4m3 K/V (per-tensor scale), bf16 Q, P16"))


def mixed_step(seed: int = 3, n_decode: int = 256, ctx_lo: int = 64, ctx_hi: int = 1024,
               prompt: int = 2662, chunk_at: int = 1024, chunk: int = 256) -> Workload:
    """n_decode decode rows plus one causal prefill chunk of `chunk` rows at
    positions chunk_at.. of a `prompt`-token prompt whose pages are reserved up
    front; Hq 16 / Hkv 8, D 128, bf16, P 32.  Rows: decode rows first, then the chunk."""
    P, Hq, Hkv, D = 32, 16, 8, 128
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=n_decode)
    max_blocks = (max(prompt, ctx_hi) + P - 1) // P
    pages = [int((L + P - 1) // P) for L in ctx] + [(prompt + P - 1) // P]
    num_pages = sum(pages) + 64
    bt = _assign_pages(rng, pages, num_pages, max_blocks)
    cs = n_decode  # the chunk's sequence id
    hist_counts = [int(L - 1) for L in ctx] + [chunk_at]
    hist_seq = np.repeat(np.arange(n_decode + 1, dtype=np.int32), hist_counts)
    hist_pos = np.concatenate([np.arange(c, dtype=np.int32) for c in hist_counts])
    hist_k, hist_v = _draw_rows(seed * 1000 + 1, hist_counts, Hkv, D, BF16)
    seq_ids = np.concatenate([np.arange(n_decode, dtype=np.int32), np.full(chunk, cs, dtype=np.int32)])
    positions = np.concatenate([(ctx - 1).astype(np.int32),
                                np.arange(chunk_at, chunk_at + chunk, dtype=np.int32)])
    n = n_decode + chunk
    q = _cast(rng.standard_normal((n, Hq, D), dtype=np.float32), BF16)
    k_new = _cast(rng.standard_normal((n, Hkv, D), dtype=np.float32), BF16)
    v_new = _cast(rng.standard_normal((n, Hkv, D), dtype=np.float32), BF16)
    return Workload(name="mixed_step", Hq=Hq, Hkv=Hkv, D=D, P=P, kv_dtype=BF16, in_dtype=BF16,
                    q_dtype=BF16, num_pages=num_pages, block_tables=bt, hist_seq=hist_seq,
                    hist_pos=hist_pos, hist_k=hist_k, hist_v=hist_v, seq_ids=seq_ids,
                    positions=positions, q=q, k_new=k_new, v_new=v_new, chunks=[(n_decode, chunk)],
                    description=f"mixed step: {n_decode} decode rows ctx U[{ctx_lo},{ctx_hi}] + one "
                                f"{chunk}-row causal prefill chunk at {chunk_at} of a {prompt}-token "
                                "prompt, Hq16/Hkv8, D128, bf16, P32, one launch")


def shared_prefix(seed: int = 4, n_seqs: int = 768, share_frac: float = 0.7, prefix: int = 90,
                  prompt: int = 128, max_gen: int = 128, P: int = 32, Hq: int = 28, Hkv: int = 4) -> Workload:
    """n_seqs sequences at position prompt + g, g ~ U{0..max_gen-1}; a fraction
    share_frac of them share a `prefix`-token prefix whose full pages are
    physically shared; Hq 28 / Hkv 4, D 128, fp8 e4m3 K/V (bf16 rows in),
    bf16 Q, P 32 by default.  The page that holds the prefix's tail is a
    private copy."""
    D = 128
    rng = np.random.Generator(np.random.PCG64(seed))
    g = rng.integers(0, max_gen, size=n_seqs)
    ctx = (prompt + g + 1).astype(np.int64)  # keys attended by each decode row
    n_share = int(round(share_frac * n_seqs))
    sharers = np.sort(rng.permutation(n_seqs)[:n_share])
    is_sharer = np.zeros(n_seqs, dtype=bool)
    is_sharer[sharers] = True
    n_shared_pages = prefix // P
    max_blocks = (prompt + max_gen + P - 1) // P
    pages_total = [int((L + P - 1) // P) for L in ctx]
    private = [pages_total[s] - (n_shared_pages if is_sharer[s] else 0) for s in range(n_seqs)]
    num_pages = n_shared_pages + sum(private) + 32
    perm = rng.permutation(num_pages).astype(np.int32)
    shared_ids = perm[:n_shared_pages]
    bt = np.full((n_seqs, max_blocks), -1, dtype=np.int32)
    k = n_shared_pages
    for s in range(n_seqs):
        j0 = 0
        if is_sharer[s]:
            bt[s, :n_shared_pages] = shared_ids
            j0 = n_shared_pages
        n = pages_total[s] - j0
        bt[s, j0:j0 + n] = perm[k:k + n]
        k += n
    # history rows: the shared pages once (through the first sharer), then each
    # sequence's own positions; sharers' tokens < prefix carry the prefix values
    kp_pre, vp_pre = _draw_rows(seed * 1000 + 7, [prefix], Hkv, D, BF16)
    first = int(sharers[0]) if n_share else -1
    own_from = [n_shared_pages * P if is_sharer[s] else 0 for s in range(n_seqs)]
    own_counts = [int(ctx[s] - 1 - own_from[s]) for s in range(n_seqs)]
    K_own, V_own = _draw_rows(seed * 1000 + 1, own_counts, Hkv, D, BF16)
    seqs, poss, Ks, Vs = [], [], [], []
    if n_share:
        m = n_shared_pages * P
        seqs.append(np.full(m, first, np.int32))
        poss.append(np.arange(m, dtype=np.int32))
        Ks.append(kp_pre[:m])
        Vs.append(vp_pre[:m])
    off = 0
    for s in range(n_seqs):
        c = own_counts[s]
        kk = K_own[off:off + c].copy()
        vv = V_own[off:off + c].copy()
        if is_sharer[s]:
            tail = prefix - own_from[s]  # prefix tokens on the private page
            kk[:tail] = kp_pre[own_from[s]:prefix]
            vv[:tail] = vp_pre[own_from[s]:prefix]
        seqs.append(np.full(c, s, np.int32))
        poss.append(np.arange(own_from[s], own_from[s] + c, dtype=np.int32))
        Ks.append(kk)
        Vs.append(vv)
        off += c
    hist_seq = np.concatenate(seqs)
    hist_pos = np.concatenate(poss)
    hist_k = np.concatenate(Ks)
    hist_v = np.concatenate(Vs)
    seq_ids = np.arange(n_seqs, dtype=np.int32)
    positions = (ctx - 1).astype(np.int32)
    q = _cast(rng.standard_normal((n_seqs, Hq, D), dtype=np.float32), BF16)
    k_new = _cast(rng.standard_normal((n_seqs, Hkv, D), dtype=np.float32), BF16)
    v_new = _cast(rng.standard_normal((n_seqs, Hkv, D), dtype=np.float32), BF16)
    # per-tensor fp8 scales: amax of every K (V) value the pools will hold, / 448, in fp32
    amax_k = max(np.abs(bf16_bits_to_f32(hist_k)).max(), np.abs(bf16_bits_to_f32(k_new)).max())
    amax_v = max(np.abs(bf16_bits_to_f32(hist_v)).max(), np.abs(bf16_bits_to_f32(v_new)).max())
    k_scale = float(np.float32(amax_k) / np.float32(448.0))
    v_scale = float(np.float32(amax_v) / np.float32(448.0))
    return Workload(name="shared_prefix", Hq=Hq, Hkv=Hkv, D=D, P=P, kv_dtype=E4M3, in_dtype=BF16,
                    q_dtype=BF16, num_pages=num_pages, block_tables=bt, hist_seq=hist_seq,
                    hist_pos=hist_pos, hist_k=hist_k, hist_v=hist_v, seq_ids=seq_ids,
                    positions=positions, q=q, k_new=k_new, v_new=v_new, k_scale=k_scale,
                    v_scale=v_scale, shared_pages=n_shared_pages if n_share > 1 else 0,
                    description=f"7B-class shared-prefix decode: batch {n_seqs}, Hq{Hq}/Hkv{Hkv}, D128, fp8 "
                                f"e4m3 K/V (per-tensor scale), bf16 Q, {prompt} prompt + U{{0..{max_gen - 1}}} "
                                f"generated, {n_share} seqs share a {prefix}-token prefix, P{P}")


def reorder_rows(wl: Workload, order) -> Workload:
    """The same decode step with its rows listed in `order` (a permutation of
    the rows): every row keeps its sequence, position, query and new K/V."""
    if wl.chunks:
        raise ValueError("reorder_rows takes decode-only steps")
    order = np.asarray(order, dtype=np.int64)
    if sorted(order.tolist()) != list(range(wl.n_rows)):
        raise ValueError("order is not a permutation of the rows")
    return replace(wl, seq_ids=wl.seq_ids[order].copy(), positions=wl.positions[order].copy(),
                   q=wl.q[order].copy(), k_new=wl.k_new[order].copy(), v_new=wl.v_new[order].copy(),
                   name=wl.name + "_grouped", description=wl.description + "; rows grouped by prefix")


def group_by_prefix(wl: Workload) -> Workload:
    """The rows listed prefix by prefix, as a scheduler that groups its batches
    by prefix would list them: rows whose sequences start on the same physical
    page become adjacent (each group in the rows' original order), groups in
    order of first appearance.  No row's inputs change."""
    first = wl.block_tables[wl.seq_ids, 0]
    _, idx_first, inv = np.unique(first, return_index=True, return_inverse=True)
    group_rank = np.argsort(np.argsort(idx_first))  # group ordinal by first appearance
    return reorder_rows(wl, np.argsort(group_rank[inv.reshape(-1)], kind="stable"))


def chunked_step(seed: int, chunks, decode_ctx=(), Hq: int = 16, Hkv: int = 8, D: int = 128, P: int = 32,
                 q_dtype: int = BF16, kv_dtype: int = BF16, spare_pages: int = 8) -> Workload:
    """Decode rows (one per context in decode_ctx) followed by prefill chunks;
    chunks = [(chunk_start, chunk_len, reserved_tokens)], one sequence each, whose
    tokens 0..chunk_start-1 are history.  Pages for reserved_tokens are taken
    up front, so the chunk's last page may hold slots past its last row."""
    rng = np.random.Generator(np.random.PCG64(seed))
    decode_ctx = [int(x) for x in decode_ctx]
    n_dec = len(decode_ctx)
    reserve = [max(L, 1) for L in decode_ctx] + [int(r) for _, _, r in chunks]
    pages = [(r + P - 1) // P for r in reserve]
    max_blocks = max(pages)
    num_pages = sum(pages) + spare_pages
    bt = _assign_pages(rng, pages, num_pages, max_blocks)
    hist_counts = [L - 1 for L in decode_ctx] + [int(c0) for c0, _, _ in chunks]
    ns = n_dec + len(chunks)
    hist_seq = np.repeat(np.arange(ns, dtype=np.int32), hist_counts)
    hist_pos = np.concatenate([np.arange(c, dtype=np.int32) for c in hist_counts]) if ns else np.zeros(0, np.int32)
    in_dtype = kv_dtype if kv_dtype != E4M3 else BF16
    hist_k, hist_v = _draw_rows(seed * 1000 + 1, hist_counts, Hkv, D, in_dtype)
    seq_ids = [np.arange(n_dec, dtype=np.int32)]
    positions = [np.array(decode_ctx, dtype=np.int32) - 1]
    spans = []
    row = n_dec
    for i, (c0, cl, _) in enumerate(chunks):
        seq_ids.append(np.full(cl, n_dec + i, dtype=np.int32))
        positions.append(np.arange(c0, c0 + cl, dtype=np.int32))
        spans.append((row, cl))
        row += cl
    seq_ids = np.concatenate(seq_ids)
    positions = np.concatenate(positions)
    n = len(seq_ids)
    q = _cast(rng.standard_normal((n, Hq, D), dtype=np.float32), q_dtype)
    k_new = _cast(rng.standard_normal((n, Hkv, D), dtype=np.float32), in_dtype)
    v_new = _cast(rng.standard_normal((n, Hkv, D), dtype=np.float32), in_dtype)
    return Workload(name="chunked", Hq=Hq, Hkv=Hkv, D=D, P=P, kv_dtype=kv_dtype, in_dtype=in_dtype, q_dtype=q_dtype,
                    num_pages=num_pages, block_tables=bt, hist_seq=hist_seq, hist_pos=hist_pos, hist_k=hist_k,
                    hist_v=hist_v, seq_ids=seq_ids, positions=positions, q=q, k_new=k_new, v_new=v_new,
                    chunks=spans, description=f"chunked step: {n_dec} decode rows + chunks {list(chunks)}")


def long_prefill(seed: int = 6, n_tokens: int = 4096, Hq: int = 16, Hkv: int = 8, D: int = 128,
                 P: int = 32) -> Workload:
    """A prefill step: one sequence's first n_tokens tokens as one causal chunk
    (no decode rows), the head shape of the mixed step."""
    wl = chunked_step(seed, [(0, n_tokens, n_tokens)], Hq=Hq, Hkv=Hkv, D=D, P=P)
    wl.name = "long_prefill"
    wl.description = (f"prefill step: one {n_tokens}-token causal chunk, Hq{Hq}/Hkv{Hkv}, D{D}, bf16, P{P}, "
                      f"no decode rows")
    return wl


CONFIGS = {
    "tiny_decode": tiny_decode,
    "batched_decode": batched_decode,
    "mixed_step": mixed_step,
    "shared_prefix": shared_prefix,
    "long_context": long_context,
    "batched_decode_fp8": batched_decode_fp8,
    "long_context_fp8": long_context_fp8,
}

# Scaled-down versions the oracle finishes in well under a second; each still
# spans several pages per sequence, a split boundary and a partial last page.
SMALL = {
    "tiny_decode": lambda: tiny_decode(),
    "batched_decode": lambda: batched_decode(n_seqs=24),
    "mixed_step": lambda: mixed_step(n_decode=16, ctx_hi=700, prompt=700, chunk_at=300, chunk=200),
    "shared_prefix": lambda: shared_prefix(n_seqs=40),
    "long_context": lambda: long_context(n_seqs=2, ctx=5000),
    "batched_decode_fp8": lambda: batched_decode_fp8(n_seqs=24),
    "long_context_fp8": lambda: long_context_fp8(n_seqs=2, ctx=5000),
}
