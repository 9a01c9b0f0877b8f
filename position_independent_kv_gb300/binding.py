"""Python binding of the C ABI in include/rk_seg_attn.h (ctypes).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of librk_seg_attn.so.  PyTorch supplies device memory and streams.
If the shared library has not been built, every entry point raises; there is
no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .build import LIB

RK_SEG_NEW = 1
RK_PLAN_HOST_ONLY = 1
RK_PLAN_LEGACY_MMA = 2
RK_PLAN_SINGLE_CTA = 4
RK_PLAN_CTA_PAIR = 8
RK_PLAN_DEVICE_BITMAP = 16
RK_PLAN_V_ROPE = 32
RK_PLAN_NO_SIDE_PAIRS = 64
RK_PROT_NONE = 1

EXPORTS = ["rk_seg_attn_plan", "rk_seg_attn_plan_destroy", "rk_seg_attn_plan_info",
           "rk_seg_attn_plan_pairs",
           "rk_seg_attn_workspace_bytes", "rk_seg_attn_forward", "rk_lse_merge",
           "rk_seg_attn_last_device_status", "rk_status_string",
           "rk_seg_attn_forward_noalloc", "rk_seg_attn_forward_host",
           "rk_protected_workspace_bytes", "rk_protected_build", "rk_project_forward",
           "rk_segpaged_plan", "rk_segpaged_forward", "rk_segpaged_plan_info",
           "rk_segpaged_last_device_status", "rk_segpaged_plan_destroy",
           "rk_segpaged_workspace_bytes"]

RK_SEGPAGED_HOST_ONLY = 1
RK_SEGPAGED_DENSE_MASK = 2

STATUS = {0: "RK_OK", 1: "RK_ERR_NULL", 2: "RK_ERR_INVALID_ARG", 3: "RK_ERR_SEGMENT_OVERLAP",
          4: "RK_ERR_SEGMENT_GAP", 5: "RK_ERR_UNSUPPORTED_DIMS", 6: "RK_ERR_CAPACITY",
          7: "RK_ERR_CUDA", 8: "RK_ERR_DEVICE_TIMEOUT", 9: "RK_ERR_PLAN_MISMATCH",
          10: "RK_ERR_ALIGNMENT", 11: "RK_ERR_WORKSPACE"}


class RkSegPagedDesc(C.Structure):
    _fields_ = [("num_requests", C.c_int32), ("seq_len", C.POINTER(C.c_int64)),
                ("q_row_begin", C.POINTER(C.c_int64)), ("num_q_heads", C.c_int32),
                ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("page_size", C.c_int32),
                ("num_pages", C.c_int64), ("max_blocks", C.c_int32),
                ("block_table", C.POINTER(C.c_int32)), ("kv_head_role", C.POINTER(C.c_uint8)),
                ("sink", C.c_int32), ("window", C.c_int32), ("softmax_scale", C.c_float),
                ("flags", C.c_uint32), ("block_delta", C.POINTER(C.c_int64)),
                ("rope_base", C.c_double)]


class RkSegPagedInfo(C.Structure):
    _fields_ = [("rows", C.c_int64), ("tiles", C.c_int64), ("pairs", C.c_int64),
                ("performed_pairs", C.c_int64), ("kv_blocks", C.c_int64),
                ("split_parts", C.c_int64), ("group", C.c_int32), ("reserved", C.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}


class RkSegment(C.Structure):
    _fields_ = [("latent", C.c_void_p), ("n", C.c_int64), ("delta", C.c_int64),
                ("flags", C.c_uint32), ("reserved", C.c_uint32)]


class RkDesc(C.Structure):
    _fields_ = [("num_requests", C.c_int32), ("seg_begin", C.POINTER(C.c_int32)),
                ("segs", C.POINTER(RkSegment)), ("q_row_begin", C.POINTER(C.c_int64)),
                ("num_heads", C.c_int32), ("d_nope", C.c_int32), ("d_rope", C.c_int32),
                ("rope_base", C.c_double), ("softmax_scale", C.c_float),
                ("head_role", C.POINTER(C.c_uint8)), ("sink", C.c_int32), ("window", C.c_int32),
                ("protected_bitmap", C.POINTER(C.c_uint32)), ("flags", C.c_uint32)]


class RkPlanInfo(C.Structure):
    _fields_ = [("rows", C.c_int64), ("num_heads", C.c_int32), ("d_nope", C.c_int32),
                ("d_rope", C.c_int32), ("num_global_heads", C.c_int32),
                ("num_local_heads", C.c_int32), ("protected_local_rows", C.c_int64),
                ("dense_tiles", C.c_int64), ("split_chunks", C.c_int64),
                ("pairs_global", C.c_int64), ("pairs_local", C.c_int64),
                ("performed_pairs", C.c_int64), ("latent_bytes", C.c_int64),
                ("kernel", C.c_int32), ("d_v", C.c_int32), ("side_pairs", C.c_int64)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


class RkProjectDesc(C.Structure):
    _fields_ = [("rows", C.c_int64), ("num_heads", C.c_int32), ("d_v", C.c_int32),
                ("d_g", C.c_int32), ("d_model", C.c_int32),
                ("head_role", C.POINTER(C.c_uint8))]


class RkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


_lib = None


def lib() -> C.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: run position_independent_kv_gb300.build.build()")
        try:
            import torch  # noqa: F401  (loads the CUDA runtime torch was built with)
        except ImportError:
            pass
        L = C.CDLL(LIB)
        L.rk_seg_attn_plan.argtypes = [C.POINTER(RkDesc), C.c_void_p, C.POINTER(C.c_void_p)]
        L.rk_seg_attn_plan.restype = C.c_int
        L.rk_seg_attn_plan_destroy.argtypes = [C.c_void_p]
        L.rk_seg_attn_plan_destroy.restype = None
        L.rk_seg_attn_plan_info.argtypes = [C.c_void_p, C.POINTER(RkPlanInfo)]
        L.rk_seg_attn_plan_info.restype = C.c_int
        L.rk_seg_attn_plan_pairs.argtypes = [C.c_void_p, C.c_void_p, C.c_int64]
        L.rk_seg_attn_plan_pairs.restype = C.c_int64
        L.rk_seg_attn_workspace_bytes.argtypes = [C.c_void_p]
        L.rk_seg_attn_workspace_bytes.restype = C.c_size_t
        L.rk_seg_attn_forward.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                          C.c_void_p, C.c_size_t, C.c_void_p]
        L.rk_seg_attn_forward.restype = C.c_int
        L.rk_project_forward.argtypes = [C.POINTER(RkProjectDesc)] + [C.c_void_p] * 9
        L.rk_project_forward.restype = C.c_int
        L.rk_protected_workspace_bytes.argtypes = [C.c_int32, C.c_int32]
        L.rk_protected_workspace_bytes.restype = C.c_size_t
        L.rk_protected_build.argtypes = [C.c_int32, C.POINTER(C.c_int32), C.POINTER(RkSegment),
                                         C.c_int32, C.c_double, C.c_int32, C.c_uint32,
                                         C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                         C.c_void_p, C.c_size_t, C.c_void_p]
        L.rk_protected_build.restype = C.c_int
        L.rk_seg_attn_forward_host.argtypes = [C.c_void_p] * 8 + [C.c_size_t, C.c_void_p]
        L.rk_seg_attn_forward_host.restype = C.c_int
        L.rk_seg_attn_forward_noalloc.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p,
                                                  C.c_void_p, C.c_void_p]
        L.rk_seg_attn_forward_noalloc.restype = C.c_int
        L.rk_lse_merge.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_int64, C.c_int32,
                                   C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]
        L.rk_lse_merge.restype = C.c_int
        L.rk_seg_attn_last_device_status.argtypes = [C.c_void_p, C.c_void_p]
        L.rk_seg_attn_last_device_status.restype = C.c_int
        L.rk_segpaged_plan.argtypes = [C.POINTER(RkSegPagedDesc), C.c_void_p,
                                       C.POINTER(C.c_void_p)]
        L.rk_segpaged_plan.restype = C.c_int
        L.rk_segpaged_forward.argtypes = [C.c_void_p] * 7 + [C.c_size_t, C.c_void_p]
        L.rk_segpaged_forward.restype = C.c_int
        L.rk_segpaged_plan_info.argtypes = [C.c_void_p, C.POINTER(RkSegPagedInfo)]
        L.rk_segpaged_plan_info.restype = C.c_int
        L.rk_segpaged_last_device_status.argtypes = [C.c_void_p, C.c_void_p]
        L.rk_segpaged_last_device_status.restype = C.c_int
        L.rk_segpaged_workspace_bytes.argtypes = [C.c_void_p]
        L.rk_segpaged_workspace_bytes.restype = C.c_size_t
        L.rk_segpaged_plan_destroy.argtypes = [C.c_void_p]
        L.rk_segpaged_plan_destroy.restype = None
        L.rk_status_string.argtypes = [C.c_int]
        L.rk_status_string.restype = C.c_char_p
        _lib = L
    return _lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(st: int, where: str):
    if st != 0:
        raise RkError(st, where)


class SegAttnPlan:
    """rk_seg_attn_plan / rk_seg_attn_forward.

    segments: list of (latent tensor or device address, n, delta, is_new)
    seg_begin: [R + 1] prefix offsets; q_row_begin: [R]
    bitmap: uint32 words per request (concatenated) or None
    """

    def __init__(self, segments, seg_begin, q_row_begin, num_heads, d_nope, d_rope,
                 rope_base, softmax_scale, head_role, sink, window, bitmap=None, flags=0,
                 stream=None):
        L = lib()
        R = len(seg_begin) - 1
        segs = (RkSegment * max(1, len(segments)))()
        for i, (lat, n, delta, is_new) in enumerate(segments):
            segs[i] = RkSegment(_ptr(lat), int(n), int(delta), RK_SEG_NEW if is_new else 0, 0)
        self._keep = [segments]
        sb = np.ascontiguousarray(seg_begin, dtype=np.int32)
        qb = np.ascontiguousarray(q_row_begin, dtype=np.int64)
        role = np.ascontiguousarray(head_role, dtype=np.uint8)
        device_bitmap = bool(flags & RK_PLAN_DEVICE_BITMAP)
        bm = (None if bitmap is None or device_bitmap
              else np.ascontiguousarray(bitmap, dtype=np.uint32))
        desc = RkDesc()
        desc.num_requests = R
        desc.seg_begin = sb.ctypes.data_as(C.POINTER(C.c_int32))
        desc.segs = segs
        desc.q_row_begin = qb.ctypes.data_as(C.POINTER(C.c_int64))
        desc.num_heads = int(num_heads)
        desc.d_nope = int(d_nope)
        desc.d_rope = int(d_rope)
        desc.rope_base = float(rope_base)
        desc.softmax_scale = float(softmax_scale)
        desc.head_role = role.ctypes.data_as(C.POINTER(C.c_uint8))
        desc.sink = int(sink)
        desc.window = int(window)
        if device_bitmap and bitmap is not None:
            desc.protected_bitmap = C.cast(C.c_void_p(_ptr(bitmap)), C.POINTER(C.c_uint32))
        else:
            desc.protected_bitmap = (bm.ctypes.data_as(C.POINTER(C.c_uint32)) if bm is not None
                                     else C.POINTER(C.c_uint32)())
        desc.flags = int(flags)
        host_only = bool(flags & RK_PLAN_HOST_ONLY)
        handle = C.c_void_p()
        st = L.rk_seg_attn_plan(C.byref(desc), 0 if host_only else _stream(stream),
                                C.byref(handle))
        _check(st, "rk_seg_attn_plan")
        self._h = handle
        self.num_heads, self.d_nope, self.d_rope = int(num_heads), int(d_nope), int(d_rope)

    @classmethod
    def from_workload(cls, wl, bitmap=None, flags=0, stream=None, addresses=None):
        from .workloads import segments_for_abi
        flat, begins = segments_for_abi(wl)
        if getattr(wl, "v_rope", False):
            flags |= RK_PLAN_V_ROPE
        if addresses is not None:
            flat = [(addresses(i, s), s[1], s[2], s[3]) for i, s in enumerate(flat)]
        return cls(flat, begins, [r.q_row_begin for r in wl.requests], wl.H, wl.d_nope,
                   wl.d_rope, wl.rope_base, wl.scale, wl.head_role, wl.sink, wl.window,
                   bitmap=bitmap, flags=flags, stream=stream)

    @property
    def info(self) -> dict:
        inf = RkPlanInfo()
        _check(lib().rk_seg_attn_plan_info(self._h, C.byref(inf)), "rk_seg_attn_plan_info")
        return inf.as_dict()

    def pairs(self):
        """rk_seg_attn_plan_pairs: int32 [n, RK_PAIR_WORDS] records of the
        4-CTA kernel's tile pairs, in the plan's order."""
        import numpy as np
        n = int(lib().rk_seg_attn_plan_pairs(self._h, None, 0))
        buf = np.zeros((max(n, 0), 20), dtype=np.int32)
        if n > 0:
            lib().rk_seg_attn_plan_pairs(self._h, buf.ctypes.data, n)
        return buf

    @property
    def workspace_bytes(self) -> int:
        return int(lib().rk_seg_attn_workspace_bytes(self._h))

    def forward(self, q, out, lse, workspace=None, stream=None):
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = lib().rk_seg_attn_forward(self._h, _ptr(q), _ptr(out), _ptr(lse), _ptr(workspace),
                                       ws_bytes, _stream(stream))
        _check(st, "rk_seg_attn_forward")

    def forward_host(self, q_host, out_host, lse_host, q, out, lse, workspace=None, stream=None):
        """rk_seg_attn_forward_host: q_host/out_host/lse_host are host tensors
        (pinned for overlap); q/out/lse are device tensors of the same shapes.
        q and lse go to the device; only the elements the kernels write come
        back into out_host (out is never uploaded)."""
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = lib().rk_seg_attn_forward_host(self._h, _ptr(q_host), _ptr(out_host), _ptr(lse_host),
                                            _ptr(q), _ptr(out), _ptr(lse), _ptr(workspace),
                                            ws_bytes, _stream(stream))
        _check(st, "rk_seg_attn_forward_host")

    def forward_noalloc(self, q, out, lse, stream=None):
        """rk_seg_attn_forward_noalloc: same results as forward, with the
        scratch in the library's static device array instead of a caller
        workspace (for callers that cannot allocate at call time)."""
        st = lib().rk_seg_attn_forward_noalloc(self._h, _ptr(q), _ptr(out), _ptr(lse),
                                               _stream(stream))
        _check(st, "rk_seg_attn_forward_noalloc")

    def device_status(self, stream=None) -> int:
        return int(lib().rk_seg_attn_last_device_status(self._h, _stream(stream)))

    def close(self):
        if getattr(self, "_h", None):
            lib().rk_seg_attn_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def lse_merge(o_parts, lse_parts, out, lse_out, stream=None):
    """rk_lse_merge: o_parts fp32 [P, rows, H, d_v], lse_parts fp32 [P, rows, H]."""
    P, rows, H, d_v = (int(x) for x in o_parts.shape)
    st = lib().rk_lse_merge(_ptr(o_parts), _ptr(lse_parts), P, rows, H, d_v, _ptr(out),
                            _ptr(lse_out), _stream(stream))
    _check(st, "rk_lse_merge")


def protected_build(segments, seg_begin, boundary, p_random, budget_pct, none, u, score, dirty,
                    bitmap, workspace, stream=None):
    """rk_protected_build.  segments: (n, delta, is_new) per segment, requests
    concatenated with prefix offsets seg_begin; u (float64), score (float32),
    dirty and bitmap (uint32 words): device tensors or None; workspace: a
    device tensor of at least protected_workspace_bytes(...) bytes."""
    segs = (RkSegment * max(1, len(segments)))()
    for i, (n, delta, is_new) in enumerate(segments):
        segs[i] = RkSegment(0, int(n), int(delta), RK_SEG_NEW if is_new else 0, 0)
    sb = np.ascontiguousarray(seg_begin, dtype=np.int32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().rk_protected_build(len(seg_begin) - 1, sb.ctypes.data_as(C.POINTER(C.c_int32)),
                                  segs, int(boundary), float(p_random), int(budget_pct),
                                  RK_PROT_NONE if none else 0, _ptr(u), _ptr(score), _ptr(dirty),
                                  _ptr(bitmap), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "rk_protected_build")


def project_forward(o, z_off, prot, w_a, w_b, z, y, head_role, status, stream=None):
    """rk_project_forward.  o bf16 [rows, H, d_v]; z_off bf16 [rows, H/8, d_g];
    prot uint32 words; w_a bf16 [H/8, d_g, 8 d_v]; w_b bf16 [d_model, H/8 d_g];
    z, y bf16 outputs; status int32 [1] (device)."""
    rows, H, dv = (int(x) for x in o.shape)
    d = RkProjectDesc()
    d.rows, d.num_heads, d.d_v = rows, H, dv
    d.d_g = int(w_a.shape[1])
    d.d_model = int(w_b.shape[0])
    role = np.ascontiguousarray(head_role, dtype=np.uint8)
    d.head_role = role.ctypes.data_as(C.POINTER(C.c_uint8))
    st = lib().rk_project_forward(C.byref(d), _ptr(o), _ptr(z_off), _ptr(prot), _ptr(w_a),
                                  _ptr(w_b), _ptr(z), _ptr(y), _ptr(status), _stream(stream))
    _check(st, "rk_project_forward")


def protected_workspace_bytes(num_requests: int, num_segments: int) -> int:
    return int(lib().rk_protected_workspace_bytes(int(num_requests), int(num_segments)))


def status_string(st: int) -> str:
    return lib().rk_status_string(int(st)).decode()


class SegPagedPlan:
    """rk_segpaged_plan / rk_segpaged_forward (SegPagedAttention on GQA).

    seq_len, q_row_begin: [R]; block_table: int32 [R, Hkv, max_blocks]
    (physical page or -1); kv_role: uint8 [Hkv] (1 = Global); block_delta:
    int64 [R, max_blocks] offsets of relocated documents, or None."""

    def __init__(self, seq_len, q_row_begin, num_q_heads, num_kv_heads, block_table, num_pages,
                 kv_role, sink, window, softmax_scale, flags=0, stream=None, head_dim=128,
                 page_size=128, block_delta=None, rope_base=10000.0):
        L = lib()
        sl = np.ascontiguousarray(seq_len, dtype=np.int64)
        qb = np.ascontiguousarray(q_row_begin, dtype=np.int64)
        tab = np.ascontiguousarray(block_table, dtype=np.int32)
        role = np.ascontiguousarray(kv_role, dtype=np.uint8)
        d = RkSegPagedDesc()
        d.num_requests = len(sl)
        d.seq_len = sl.ctypes.data_as(C.POINTER(C.c_int64))
        d.q_row_begin = qb.ctypes.data_as(C.POINTER(C.c_int64))
        d.num_q_heads = int(num_q_heads)
        d.num_kv_heads = int(num_kv_heads)
        d.head_dim = int(head_dim)
        d.page_size = int(page_size)
        d.num_pages = int(num_pages)
        d.max_blocks = int(tab.shape[-1])
        d.block_table = tab.ctypes.data_as(C.POINTER(C.c_int32))
        d.kv_head_role = role.ctypes.data_as(C.POINTER(C.c_uint8))
        d.sink = int(sink)
        d.window = int(window)
        d.softmax_scale = float(softmax_scale)
        d.flags = int(flags)
        dl = None
        if block_delta is not None:
            dl = np.ascontiguousarray(block_delta, dtype=np.int64)
            assert dl.shape == (len(sl), tab.shape[-1])
            d.block_delta = dl.ctypes.data_as(C.POINTER(C.c_int64))
        d.rope_base = float(rope_base)
        handle = C.c_void_p()
        host_only = bool(flags & RK_SEGPAGED_HOST_ONLY)
        _check(L.rk_segpaged_plan(C.byref(d), 0 if host_only else _stream(stream),
                                  C.byref(handle)), "rk_segpaged_plan")
        self._h = handle

    @classmethod
    def from_workload(cls, pw, flags=0, stream=None):
        return cls(pw.seq_len, pw.q_row_begin, pw.Hq, pw.Hkv, pw.block_table, pw.num_pages,
                   pw.kv_role, pw.sink, pw.window, pw.scale, flags=flags, stream=stream,
                   block_delta=pw.block_delta, rope_base=pw.rope_base)

    @property
    def info(self) -> dict:
        inf = RkSegPagedInfo()
        _check(lib().rk_segpaged_plan_info(self._h, C.byref(inf)), "rk_segpaged_plan_info")
        return inf.as_dict()

    @property
    def workspace_bytes(self) -> int:
        return int(lib().rk_segpaged_workspace_bytes(self._h))

    def forward(self, q, k_pages, v_pages, out, lse, workspace=None, stream=None):
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(lib().rk_segpaged_forward(self._h, _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                         _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                         _stream(stream)), "rk_segpaged_forward")

    def device_status(self, stream=None) -> int:
        return int(lib().rk_segpaged_last_device_status(self._h, _stream(stream)))

    def close(self):
        if getattr(self, "_h", None):
            lib().rk_segpaged_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
