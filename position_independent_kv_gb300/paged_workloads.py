"""Seeded synthetic inputs for SegPagedAttention on grouped-query attention.

This module only draws numbers and lays out pages; it holds none of the
method's arithmetic (no masking, no softmax).  The CUDA path and the CPU
oracle both consume what it returns.

Shapes follow the RedKnot blog ("RedKnot, explained", "Insight 3"): a model
"shaped like Qwen3-32B" -- 64 query heads over 8 KV heads of dimension 128 --
with its KV cache stored per KV head in pages; one KV head in eight is
Global, the rest Local with the MLA workloads' sink 4 and window 256 (the
blog's worked example).  A page holds 128 tokens of one KV head; the physical
pages of all (request, KV head, block) triples are a seeded permutation of
the page pool.  Where `local_pages_only` is set (decode steps), a Local head
keeps only the pages of its sink and its window, the memory claim of the
blog; the others are absent (-1) and not allocated.

Relocated documents (`docs` > 0): the first whole pages of each prompt are
split into `docs` documents of seeded page-multiple lengths (a fixed length
when `doc_tokens` is set); each was cached alone, so its keys carry their RoPE
at positions 0..n-1, and `block_delta[r, b]` holds the offset of the document
of block b (0 for the blocks after the documents).  Only the offsets are
drawn here; the keys themselves are i.i.d. as for the other workloads.

Tensors: q bf16 [rows, Hq, 128] (RoPE already at absolute positions),
k_pages / v_pages bf16 [pages, 128, 128], out bf16 [rows, Hq, 128], lse fp32
[rows, Hq].  Values are i.i.d. N(0, 1) / sqrt(128) drawn in fp32 and cast to
bf16; q_scale multiplies the queries (a sharper softmax for tests).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

PAGE = 128
HEAD_DIM = 128


@dataclass
class PagedSpec:
    name: str
    Hq: int
    Hkv: int
    seq_len: list[int]
    q_row_begin: list[int]          # per request; -1 = the last row (decode)
    sink: int = 4
    window: int = 256
    global_every: int = 8           # KV head g is Global when g % global_every == global_every - 1
    local_pages_only: bool = False
    docs: int = 0                   # relocated documents per prompt (0: none)
    doc_tokens: int = 0             # fixed document length (0: seeded page multiples)


PAGED_SPECS: dict[str, PagedSpec] = {
    # one 128K-token prefill, Qwen3-32B shape
    "qwen32b_128k": PagedSpec("qwen32b_128k", 64, 8, [131072], [0]),
    # a 16K-token version for profiling captures
    "qwen32b_16k": PagedSpec("qwen32b_16k", 64, 8, [16384], [0]),
    # 64 decode steps over 8K-64K tokens: Local heads keep sink + window pages
    "qwen32b_decode": PagedSpec("qwen32b_decode", 64, 8, [], [], local_pages_only=True),
    # reduced versions the oracle evaluates on every row; ragged last blocks,
    # several group sizes, Global and Local heads
    "paged_mini": PagedSpec("paged_mini", 16, 2, [1000, 333], [0, 200], global_every=2),
    "paged_mini_g4": PagedSpec("paged_mini_g4", 16, 4, [777], [0], global_every=2),
    "paged_mini_g1": PagedSpec("paged_mini_g1", 4, 4, [530], [0], global_every=4),
    "paged_mini_g16": PagedSpec("paged_mini_g16", 32, 2, [650], [0], global_every=2),
    "paged_decode_mini": PagedSpec("paged_decode_mini", 16, 2, [], [], global_every=2,
                                   local_pages_only=True),
    # decode rows over 8.5K-12K tokens: the Global heads' walks are split
    "paged_decode_long_mini": PagedSpec("paged_decode_long_mini", 16, 2, [], [],
                                        global_every=2, local_pages_only=True),
    # decode steps of other group sizes: 16 query pairs (every row of the
    # decode kernel's fragments), one pair, four pairs
    "paged_decode_g16_long": PagedSpec("paged_decode_g16_long", 32, 2, [], [], global_every=2,
                                       local_pages_only=True),
    "paged_decode_g1_long": PagedSpec("paged_decode_g1_long", 4, 4, [], [], global_every=4,
                                      local_pages_only=True),
    "paged_decode_g4": PagedSpec("paged_decode_g4", 8, 2, [], [], global_every=2,
                                 local_pages_only=True),
    # prefills whose last tile has at most 16 query pairs over several rows
    # (13 rows x G 1, 7 rows x G 2), and 4 rows x G 4 at the end of a 7K
    # prompt (a Global walk of 55 blocks split in two parts)
    "paged_tail_g1": PagedSpec("paged_tail_g1", 2, 2, [525], [0], global_every=2),
    "paged_tail_g2": PagedSpec("paged_tail_g2", 4, 2, [391], [0], global_every=2),
    "paged_tail_g4_split": PagedSpec("paged_tail_g4_split", 8, 2, [7000], [6996], global_every=2),
    # relocated documents (keys cached at canonical positions, the query
    # turns by -delta): several group sizes, ragged tails, decode rows
    "paged_reloc_mini": PagedSpec("paged_reloc_mini", 16, 2, [1000, 700], [0, 300],
                                  global_every=2, docs=3),
    "paged_reloc_g8": PagedSpec("paged_reloc_g8", 64, 8, [900], [0], docs=4),
    "paged_reloc_g1": PagedSpec("paged_reloc_g1", 4, 4, [530], [0], global_every=4, docs=2),
    "paged_reloc_decode": PagedSpec("paged_reloc_decode", 16, 2, [], [], global_every=2,
                                    local_pages_only=True, docs=3),
    # the 128K prefill with its first 96K tokens as 48 relocated documents of
    # 2048 tokens (the MLA long-context geometry's documents) and a 32K tail
    "qwen32b_reloc_128k": PagedSpec("qwen32b_reloc_128k", 64, 8, [131072], [0], docs=48,
                                    doc_tokens=2048),
}


@dataclass
class PagedWorkload:
    name: str
    Hq: int
    Hkv: int
    seq_len: np.ndarray          # int64 [R]
    q_row_begin: np.ndarray      # int64 [R]
    kv_role: np.ndarray          # uint8 [Hkv]
    block_table: np.ndarray      # int32 [R, Hkv, max_blocks]
    num_pages: int
    sink: int
    window: int
    block_delta: np.ndarray | None = None   # int64 [R, max_blocks] document offsets, or None
    rope_base: float = 10000.0
    q: torch.Tensor | None = None
    k_pages: torch.Tensor | None = None
    v_pages: torch.Tensor | None = None

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(HEAD_DIM)

    @property
    def rows(self) -> int:
        return int((self.seq_len - self.q_row_begin).sum())

    def row_offsets(self) -> list[int]:
        out, acc = [], 0
        for T, qb in zip(self.seq_len, self.q_row_begin):
            out.append(acc)
            acc += int(T - qb)
        return out


def _decode_lengths(name: str, rng: np.random.Generator):
    if name == "qwen32b_decode":
        return [int(x) for x in rng.integers(8192, 65537, size=64)]
    if name.endswith("_long_mini") or name.endswith("_long"):
        return [int(x) for x in rng.integers(8500, 12001, size=3)]
    return [int(x) for x in rng.integers(300, 1501, size=5)]


def make_paged_geometry(name: str, seed: int = 0) -> PagedWorkload:
    sp = PAGED_SPECS[name]
    rng = np.random.default_rng(seed)
    if sp.seq_len:
        lens = list(sp.seq_len)
        qbs = [qb if qb >= 0 else T - 1 for T, qb in zip(lens, sp.q_row_begin)]
    else:
        lens = _decode_lengths(name, rng)
        qbs = [T - 1 for T in lens]
    role = np.zeros(sp.Hkv, np.uint8)
    role[sp.global_every - 1::sp.global_every] = 1
    R = len(lens)
    max_blocks = max((T + PAGE - 1) // PAGE for T in lens)
    table = np.full((R, sp.Hkv, max_blocks), -1, np.int32)
    keep = []
    for r, T in enumerate(lens):
        nb = (T + PAGE - 1) // PAGE
        for g in range(sp.Hkv):
            blocks = range(nb)
            if sp.local_pages_only and not role[g]:
                # the pages the decode row can see: the sink's and the window's
                lo = max(0, qbs[r] - sp.window) // PAGE
                sb = (min(sp.sink, T) + PAGE - 1) // PAGE
                blocks = sorted(set(range(sb)) | set(range(lo, nb)))
            for b in blocks:
                keep.append((r, g, b))
    perm = rng.permutation(len(keep))
    for i, (r, g, b) in enumerate(keep):
        table[r, g, b] = int(perm[i])
    delta = None
    if sp.docs:
        delta = np.zeros((R, max_blocks), np.int64)
        for r, T in enumerate(lens):
            if sp.doc_tokens:
                nb_docs = min(sp.docs * sp.doc_tokens, T) // PAGE
                cuts = [d * (sp.doc_tokens // PAGE) for d in range(sp.docs) if
                        d * (sp.doc_tokens // PAGE) < nb_docs]
            else:
                nb_docs = max(0, T // PAGE - 1)   # whole pages, the last one left to the tail
                nd = min(sp.docs, nb_docs)
                cuts = ([0] + sorted(rng.choice(np.arange(1, nb_docs), size=nd - 1,
                                                replace=False).tolist()) if nd > 1 else [0])
            for i, c in enumerate(cuts):
                e = cuts[i + 1] if i + 1 < len(cuts) else nb_docs
                delta[r, c:e] = c * PAGE
    return PagedWorkload(name=name, Hq=sp.Hq, Hkv=sp.Hkv, seq_len=np.array(lens, np.int64),
                         q_row_begin=np.array(qbs, np.int64), kv_role=role, block_table=table,
                         num_pages=len(keep), sink=sp.sink, window=sp.window, block_delta=delta)


def _randn_bf16(shape, gen, device, std, chunk=4096):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for s in range(0, shape[0], chunk):
        e = min(shape[0], s + chunk)
        t = torch.randn((e - s,) + tuple(shape[1:]), generator=gen, device=device,
                        dtype=torch.float32)
        out[s:e] = (t * std).to(torch.bfloat16)
    return out


def make_paged_workload(name: str, seed: int = 0, device="cpu", q_scale: float = 1.0):
    """Geometry plus seeded bf16 tensors on `device`."""
    pw = make_paged_geometry(name, seed)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1000003 + 41)
    std = 1.0 / math.sqrt(HEAD_DIM)
    pw.k_pages = _randn_bf16((pw.num_pages, PAGE, HEAD_DIM), gen, device, std)
    pw.v_pages = _randn_bf16((pw.num_pages, PAGE, HEAD_DIM), gen, device, std)
    pw.q = _randn_bf16((pw.rows, pw.Hq, HEAD_DIM), gen, device, std * q_scale)
    return pw
