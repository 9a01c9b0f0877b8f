"""Seeded synthetic inputs for segment-relocated MLA attention.

This module only draws numbers and lays out geometry; it holds none of the
method's arithmetic (no rotation, no masking, no softmax, no protected-set
rule).  Both the CUDA path and the CPU oracle consume what it returns, so the
two sides see identical inputs.

Workloads follow the RedKnot-MLA paper (arXiv 2609.07008): per-document
latent caches built at positions 0..n-1 and placed at request offsets, a
Local/Global head split with one Global head in every group of eight
(section on the Flash/Pro profiles), sink + window for Local heads (RedKnot
blog, "Insight 1"), and a protected-row set made of query/new rows, segment
boundary rows and extra rows (paper, protected-set paragraph).  The random
numbers that the protected-set rule consumes (one uniform per row and one
permutation of the rows) are drawn here and passed in, so the rule itself can
live with the method and with the oracle independently.

Tensor conventions
------------------
latent  bf16 [n, d_nope + d_rope]  row = [c_nope | k_rope], k_rope rotated at
        the row's canonical position 0..n-1 (interleaved pairs).
q       bf16 [rows, H, d_nope + d_rope]  q_rope rotated at the row's absolute
        request position.
out     bf16 [rows, H, d_v]  pre-filled with the cached Local values; d_v =
        d_nope, or d_k for the workloads whose value carries a rotary part
        (`v_rope`: V is the whole latent row).
lse     fp32 [rows, H]  pre-filled with LSE_SENTINEL.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

LSE_SENTINEL = 12345.0


@dataclass
class Segment:
    doc: int            # index of the document (order in the latent pool)
    n: int              # rows
    delta: int          # request offset of row 0
    is_new: bool        # the request's own new rows (causal within)
    latent: torch.Tensor | None = None   # bf16 [n, d_k]


@dataclass
class Request:
    segments: list[Segment]          # table order (== document order)
    T: int                           # total rows of the request
    q_row_begin: int                 # first computed row (absolute position)
    u: np.ndarray | None = None      # float64 [T] uniforms for the protected rule
    perm: np.ndarray | None = None   # int64 [T] permutation for the protected rule

    @property
    def n_computed(self) -> int:
        return self.T - self.q_row_begin


@dataclass
class ProtectRule:
    """Parameters of the protected-row rule (the rule itself is not here)."""
    boundary: int = 128        # first/last rows of each cached segment
    p_random: float = 0.0      # independent Bernoulli probability per cached row
    budget: float = 0.0        # fraction of cached rows to reach (boundary first)
    none: bool = False         # only the query/new rows


@dataclass
class Workload:
    name: str
    H: int
    d_nope: int
    d_rope: int
    rope_base: float
    sink: int
    window: int
    head_role: np.ndarray                  # uint8 [H], 1 = Global
    requests: list[Request]
    rule: ProtectRule
    q: torch.Tensor | None = None          # bf16 [rows, H, d_k]
    out_init: torch.Tensor | None = None   # bf16 [rows, H, d_v]
    lse_init: torch.Tensor | None = None   # fp32 [rows, H]
    latent_pool: torch.Tensor | None = None
    notes: dict = field(default_factory=dict)
    v_rope: bool = False                   # V = the whole latent row (d_v = d_k)

    @property
    def d_k(self) -> int:
        return self.d_nope + self.d_rope

    @property
    def d_v(self) -> int:
        return self.d_k if self.v_rope else self.d_nope

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_k)

    @property
    def rows(self) -> int:
        return sum(r.n_computed for r in self.requests)

    def row_offsets(self) -> list[int]:
        off, acc = [], 0
        for r in self.requests:
            off.append(acc)
            acc += r.n_computed
        return off


# --------------------------------------------------------------------------
# geometry specs
# --------------------------------------------------------------------------

def _roles(H: int) -> np.ndarray:
    role = np.zeros(H, dtype=np.uint8)
    role[7::8] = 1            # head 8g+7 is the Global head of group g
    return role


@dataclass
class Spec:
    name: str
    H: int
    d_nope: int
    d_rope: int
    sink: int
    window: int
    rule: ProtectRule
    seg_lengths: list[int] | None = None     # fixed lengths (prefill)
    seg_len_range: tuple[int, int] | None = None
    n_segments: int = 0
    n_new: int = 0
    shuffle: bool = True
    outlier_frac: float = 0.0
    decode_requests: int = 0
    decode_len_range: tuple[int, int] = (0, 0)
    decode_seg_range: tuple[int, int] = (0, 0)
    rope_base: float = 10000.0
    v_rope: bool = False
    q_tail: int = 0          # prefill: compute only the last q_tail rows (0 = all)


SPECS: dict[str, Spec] = {
    # the five workloads of the benchmark
    "tiny": Spec("tiny", 8, 128, 32, 4, 64, ProtectRule(boundary=16),
                 seg_lengths=[256, 256], n_new=64, shuffle=False),
    "flash": Spec("flash", 64, 512, 64, 4, 256, ProtectRule(boundary=128, p_random=0.10),
                  seg_lengths=[4096] * 8, n_new=1024),
    "varlen": Spec("varlen", 64, 512, 64, 4, 256, ProtectRule(boundary=128, budget=0.20),
                   seg_len_range=(512, 8192), n_segments=24, n_new=4096, outlier_frac=0.01),
    "ctx128k": Spec("ctx128k", 128, 512, 64, 4, 256, ProtectRule(boundary=128, budget=0.25),
                    seg_lengths=[2048] * 48, n_new=32768),
    "decode": Spec("decode", 64, 512, 64, 4, 256, ProtectRule(none=True),
                   decode_requests=64, decode_len_range=(8192, 65536), decode_seg_range=(4, 32)),
    # reduced versions that the oracle evaluates on every row in seconds; they
    # keep the head counts, dims and rules and still span several tiles with
    # ragged tails
    "flash_mini": Spec("flash_mini", 64, 512, 64, 4, 256, ProtectRule(boundary=24, p_random=0.10),
                       seg_lengths=[300, 257, 190], n_new=77),
    "varlen_mini": Spec("varlen_mini", 64, 512, 64, 4, 256, ProtectRule(boundary=24, budget=0.20),
                        seg_len_range=(40, 300), n_segments=5, n_new=100, outlier_frac=0.01),
    "ctx128k_mini": Spec("ctx128k_mini", 128, 512, 64, 4, 256, ProtectRule(boundary=24, budget=0.25),
                         seg_lengths=[130] * 5, n_new=203),
    "decode_mini": Spec("decode_mini", 64, 512, 64, 4, 256, ProtectRule(none=True),
                        decode_requests=5, decode_len_range=(300, 1500), decode_seg_range=(2, 6)),
    # a 16K-row version of the long-context workload for profiling captures
    # (inputs larger than L2, a few GB on the device)
    "ctx16k": Spec("ctx16k", 128, 512, 64, 4, 256, ProtectRule(boundary=128, budget=0.25),
                   seg_lengths=[2048] * 6, n_new=4096),
    # the long-context geometry with only its last 2048 rows computed: the
    # longest causal tiles (the steady state of the full workload) in a
    # capture of a few GB
    "ctx128k_tail2k": Spec("ctx128k_tail2k", 128, 512, 64, 4, 256,
                           ProtectRule(boundary=128, budget=0.25),
                           seg_lengths=[2048] * 48, n_new=32768, q_tail=2048),
    "ctx128k_vrope_tail2k": Spec("ctx128k_vrope_tail2k", 128, 448, 64, 4, 256,
                                 ProtectRule(boundary=128, budget=0.25),
                                 seg_lengths=[2048] * 48, n_new=32768, q_tail=2048, v_rope=True),
    "tiny_wide": Spec("tiny_wide", 8, 128, 32, 4, 10000, ProtectRule(boundary=16),
                      seg_lengths=[256, 256], n_new=64, shuffle=False),
    # degenerate cases of the method: no sink and a zero window (a Local row
    # sees only itself), one-row segments, decode requests of a few rows,
    # the smallest head count, many short segments with one row per Local tile
    "edge_sink0_w0": Spec("edge_sink0_w0", 64, 512, 64, 0, 0, ProtectRule(boundary=8, p_random=0.5),
                          seg_lengths=[37, 1, 64], n_new=5),
    "edge_tiny_decode": Spec("edge_tiny_decode", 64, 512, 64, 4, 256, ProtectRule(none=True),
                             decode_requests=6, decode_len_range=(1, 9), decode_seg_range=(1, 3)),
    "edge_h8": Spec("edge_h8", 8, 512, 64, 4, 16, ProtectRule(boundary=4, budget=0.25),
                    seg_lengths=[40, 75], n_new=13),
    "edge_many_segs": Spec("edge_many_segs", 128, 512, 64, 2, 7, ProtectRule(boundary=1, budget=0.10),
                           seg_len_range=(1, 9), n_segments=40, n_new=30),
    # a value that carries a rotary part (V = the whole latent row, output
    # phase restored): the long-context and decode geometries with a 512-wide
    # latent row of 448 nope + 64 rope dims, and reduced versions for parity
    "ctx128k_vrope": Spec("ctx128k_vrope", 128, 448, 64, 4, 256,
                          ProtectRule(boundary=128, budget=0.25),
                          seg_lengths=[2048] * 48, n_new=32768, v_rope=True),
    "decode_vrope": Spec("decode_vrope", 64, 448, 64, 4, 256, ProtectRule(none=True),
                         decode_requests=64, decode_len_range=(8192, 65536),
                         decode_seg_range=(4, 32), v_rope=True),
    "ctx16k_vrope": Spec("ctx16k_vrope", 128, 448, 64, 4, 256,
                         ProtectRule(boundary=128, budget=0.25),
                         seg_lengths=[2048] * 6, n_new=4096, v_rope=True),
    "flash_vrope_mini": Spec("flash_vrope_mini", 64, 448, 64, 4, 256,
                             ProtectRule(boundary=24, p_random=0.10),
                             seg_lengths=[300, 257, 190], n_new=77, v_rope=True),
    "ctx128k_vrope_mini": Spec("ctx128k_vrope_mini", 128, 448, 64, 4, 256,
                               ProtectRule(boundary=24, budget=0.25),
                               seg_lengths=[130] * 5, n_new=203, v_rope=True),
    "decode_vrope_mini": Spec("decode_vrope_mini", 64, 448, 64, 4, 256, ProtectRule(none=True),
                              decode_requests=5, decode_len_range=(300, 1500),
                              decode_seg_range=(2, 6), v_rope=True),
}


def _composition(rng: np.random.Generator, total: int, parts: int) -> list[int]:
    """Random composition of `total` into `parts` positive integers."""
    cuts = np.sort(rng.choice(np.arange(1, total), size=parts - 1, replace=False))
    edges = np.concatenate([[0], cuts, [total]])
    return [int(x) for x in np.diff(edges)]


def make_geometry(name: str, seed: int = 0) -> Workload:
    """Segment tables, roles and the protected-rule draws (no tensors yet)."""
    spec = SPECS[name]
    rng = np.random.default_rng(seed)
    requests: list[Request] = []
    if spec.decode_requests:
        lo, hi = spec.decode_len_range
        slo, shi = spec.decode_seg_range
        doc = 0
        for _ in range(spec.decode_requests):
            L = int(rng.integers(lo, hi + 1))
            S = min(int(rng.integers(slo, shi + 1)), L)   # at least one row per segment
            lens = _composition(rng, L, S)
            order = rng.permutation(S)
            segs = []
            pos = 0
            deltas = [0] * S
            for j in order:
                deltas[j] = pos
                pos += lens[j]
            for j in range(S):
                segs.append(Segment(doc=doc, n=lens[j], delta=deltas[j], is_new=False))
                doc += 1
            segs.append(Segment(doc=doc, n=1, delta=L, is_new=True))
            doc += 1
            requests.append(Request(segments=segs, T=L + 1, q_row_begin=L))
    else:
        if spec.seg_lengths is not None:
            lens = list(spec.seg_lengths)
        else:
            a, b = spec.seg_len_range
            lens = [int(x) for x in rng.integers(a, b + 1, size=spec.n_segments)]
        S = len(lens)
        order = rng.permutation(S) if spec.shuffle else np.arange(S)
        deltas = [0] * S
        pos = 0
        for j in order:
            deltas[j] = pos
            pos += lens[j]
        segs = [Segment(doc=j, n=lens[j], delta=deltas[j], is_new=False) for j in range(S)]
        segs.append(Segment(doc=S, n=spec.n_new, delta=pos, is_new=True))
        T = pos + spec.n_new
        qb = T - spec.q_tail if spec.q_tail else 0
        requests.append(Request(segments=segs, T=T, q_row_begin=qb))
    for req in requests:
        req.u = rng.random(req.T)
        req.perm = rng.permutation(req.T).astype(np.int64)
    return Workload(name=name, H=spec.H, d_nope=spec.d_nope, d_rope=spec.d_rope,
                    rope_base=spec.rope_base, sink=spec.sink, window=spec.window,
                    head_role=_roles(spec.H), requests=requests, rule=spec.rule,
                    v_rope=spec.v_rope)


def _randn_bf16(shape, gen: torch.Generator, device, std: float, chunk_rows: int = 2048) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 and cast to bf16, generated in row chunks."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    n = shape[0]
    for s in range(0, n, chunk_rows):
        e = min(n, s + chunk_rows)
        t = torch.randn((e - s,) + tuple(shape[1:]), generator=gen, device=device, dtype=torch.float32)
        out[s:e] = (t * std).to(torch.bfloat16)
    return out


def make_workload(name: str, seed: int = 0, device: str | torch.device = "cpu",
                  q_scale: float = 1.0, with_out: bool = True) -> Workload:
    """Full workload: geometry plus seeded bf16 tensors on `device`.

    Latents and queries are i.i.d. N(0,1)/sqrt(d_k); `q_scale` multiplies the
    queries (a sharper softmax for tests).  Outlier rows (varlen) are scaled
    by 8 before the bf16 cast.  The pre-filled output comes from a second
    generator stream of the same seed.
    """
    wl = make_geometry(name, seed)
    spec = SPECS[name]
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1000003 + 17)
    std = 1.0 / math.sqrt(wl.d_k)
    total_lat = sum(s.n for r in wl.requests for s in r.segments)
    pool = _randn_bf16((total_lat, wl.d_k), gen, device, std)
    if spec.outlier_frac > 0:
        rs = np.random.default_rng(seed + 7)
        mask = rs.random(total_lat) < spec.outlier_frac
        idx = torch.from_numpy(np.nonzero(mask)[0]).to(device)
        if idx.numel():
            pool[idx] = (pool[idx].float() * 8.0).to(torch.bfloat16)
        wl.notes["outlier_rows"] = int(mask.sum())
    # carve per-segment views in document order
    off = 0
    for r in wl.requests:
        for s in r.segments:
            s.latent = pool[off:off + s.n]
            off += s.n
    wl.latent_pool = pool
    wl.q = _randn_bf16((wl.rows, wl.H, wl.d_k), gen, device, std * q_scale)
    if with_out:
        gen2 = torch.Generator(device=device)
        gen2.manual_seed(seed * 1000003 + 29)
        wl.out_init = _randn_bf16((wl.rows, wl.H, wl.d_v), gen2, device, 1.0)
        wl.lse_init = torch.full((wl.rows, wl.H), LSE_SENTINEL, dtype=torch.float32, device=device)
    return wl


def segments_for_abi(wl: Workload):
    """Flattened (latent tensor, n, delta, is_new) list and per-request begins."""
    flat, begins = [], [0]
    for r in wl.requests:
        for s in r.segments:
            flat.append((s.latent, s.n, s.delta, s.is_new))
        begins.append(len(flat))
    return flat, begins
