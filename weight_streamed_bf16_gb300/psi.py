"""ctypes binding of libpsi (include/psi.h): the same entry points, argument
marshalling only.  Every step of the operators runs in the library's CUDA
kernels; there is no Python or CPU fallback.  Loading fails loudly when the
library has not been built.

Pointers are passed as Python ints (device or pinned-host addresses, e.g.
``tensor.data_ptr()``); streams as ints (``torch.cuda.Stream.cuda_stream``).
Each wrapper raises ``PsiError`` when the library returns a non-OK status.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpsi.so")

PSI_OK = 0
PSI_ERR_INVALID_ARG = 1
PSI_ERR_CAPACITY = 2
PSI_ERR_PAGE_BUSY = 3
PSI_ERR_CUDA = 4
PSI_ERR_TIMEOUT = 5
PSI_ERR_UNSUPPORTED = 6
PSI_ERR_DEVICE = 7

PSI_RESIDENT = 0x1
PSI_SYNC_COPY = 0x2
PSI_BOUNDARY_PREGELU_BF16 = 0x4
PSI_BIAS_AFTER_BF16 = 0x8
PSI_ATTN_BF16_WEIGHTS = 0x10
PSI_ROPE_AFTER_BF16 = 0x20

# every entry point include/psi.h declares
EXPORTS = [
    "psi_version", "psi_status_string", "psi_last_error",
    "psi_plan_linear", "psi_plan_columns", "psi_ffn_page_bytes", "psi_ffn_pack", "psi_ffn_workspace",
    "psi_arena_create", "psi_arena_destroy", "psi_arena_slots",
    "psi_page_stream", "psi_page_release", "psi_sync", "psi_stream_wait",
    "psi_arena_stats", "psi_arena_reset_stats", "psi_arena_set_timing", "psi_kernel_launches",
    "psi_arena_trace_begin", "psi_arena_trace_get",
    "psi_arena_fail_next_copy", "psi_debug_stall_next_gemm",
    "psi_linear_paged", "psi_linear_rope_paged", "psi_rmsnorm",
    "psi_ffn_paged", "psi_ffn_paged_strided", "psi_attn_partitioned", "psi_attn_partitioned_ws",
    "psi_attn_workspace_size",
    "psi_ffn_resident_noalloc",
    "psi_journal_create", "psi_journal_destroy", "psi_journal_commit", "psi_journal_reload",
    "psi_journal_acquire", "psi_journal_fence", "psi_journal_drop", "psi_journal_host_view",
    "psi_journal_get_stats", "psi_journal_fail_next_copy",
]


class PsiError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_status_name(status)}: {msg}")
        self.status = status


class psi_page(C.Structure):
    _fields_ = [("slot", C.c_int32), ("seq", C.c_uint64), ("dev", C.c_void_p),
                ("bytes", C.c_size_t)]


class psi_linear_weight(C.Structure):
    _fields_ = [("host", C.c_void_p), ("dev_resident", C.c_void_p), ("rows", C.c_int64),
                ("cols", C.c_int64), ("page_rows", C.c_int64)]


class psi_ffn_weight(C.Structure):
    _fields_ = [("host", C.c_void_p), ("dev_resident", C.c_void_p), ("d", C.c_int64),
                ("h", C.c_int64), ("r", C.c_int64), ("slice", C.c_int64)]


class psi_rope(C.Structure):
    _fields_ = [("cos", C.c_void_p), ("sin", C.c_void_p), ("ld", C.c_int64),
                ("cols", C.c_int64), ("dh", C.c_int32), ("pad_", C.c_int32)]


class psi_key(C.Structure):
    _fields_ = [("block", C.c_int32), ("branch", C.c_int32), ("role", C.c_int32)]


class psi_journal_stats(C.Structure):
    _fields_ = [("commits", C.c_uint64), ("reloads", C.c_uint64), ("d2h_bytes", C.c_uint64),
                ("h2d_bytes", C.c_uint64), ("host_waits", C.c_uint64),
                ("hazard_waits", C.c_uint64), ("slots_in_use", C.c_int32),
                ("slots_total", C.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class psi_heads(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("ld_token", C.c_int64), ("ld_head", C.c_int64)]


class psi_stats(C.Structure):
    _fields_ = [("pages_streamed", C.c_uint64), ("h2d_bytes", C.c_uint64),
                ("resident_pages", C.c_uint64), ("kernels_launched", C.c_uint64),
                ("timed_gemms", C.c_uint64), ("gemm_ms", C.c_double),
                ("gemm_flops", C.c_double), ("timed_copies", C.c_uint64),
                ("copy_ms", C.c_double), ("copy_bytes", C.c_double),
                ("gemm_busy_ms", C.c_double), ("copy_busy_ms", C.c_double)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


PSI_TRACE_COPY = 0
PSI_TRACE_GEMM = 1


class psi_trace_record(C.Structure):
    _fields_ = [("kind", C.c_int32), ("slot", C.c_int32), ("stream", C.c_int32),
                ("pad_", C.c_int32), ("seq", C.c_uint64), ("start_ms", C.c_double),
                ("end_ms", C.c_double), ("work", C.c_double)]

    def as_dict(self):
        return {"kind": "copy" if self.kind == PSI_TRACE_COPY else "gemm", "slot": self.slot,
                "stream": self.stream, "seq": self.seq, "start_ms": self.start_ms,
                "end_ms": self.end_ms, "work": self.work}


_lib = None


def _status_name(s):
    names = {0: "PSI_OK", 1: "PSI_ERR_INVALID_ARG", 2: "PSI_ERR_CAPACITY",
             3: "PSI_ERR_PAGE_BUSY", 4: "PSI_ERR_CUDA", 5: "PSI_ERR_TIMEOUT",
             6: "PSI_ERR_UNSUPPORTED", 7: "PSI_ERR_DEVICE"}
    return names.get(s, f"status {s}")


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libpsi.so (raises if it is missing: build it with build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libpsi.so not found at {path}; run "
                           "weight_streamed_bf16_gb300.build.build() (needs nvcc)")
    lib = C.CDLL(path)
    vp, i32, i64, u32, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_uint32, C.c_size_t
    st = C.c_int
    sig = {
        "psi_version": (C.c_char_p, []),
        "psi_status_string": (C.c_char_p, [st]),
        "psi_last_error": (C.c_char_p, []),
        "psi_plan_linear": (st, [i64, i64, sz, C.POINTER(i64)]),
        "psi_plan_columns": (st, [i64, i64, i32, i32, C.POINTER(i64), C.POINTER(i64)]),
        "psi_ffn_page_bytes": (sz, [i64, i64, i64]),
        "psi_ffn_pack": (st, [vp, vp, i64, i64, i64, i64, vp]),
        "psi_ffn_workspace": (st, [i64, i64, i64, C.POINTER(sz), C.POINTER(sz)]),
        "psi_arena_create": (st, [vp, sz, sz, vp, vp, C.POINTER(vp)]),
        "psi_arena_destroy": (st, [vp]),
        "psi_arena_slots": (i32, [vp]),
        "psi_page_stream": (st, [vp, vp, sz, u32, C.POINTER(psi_page)]),
        "psi_page_release": (st, [vp, psi_page]),
        "psi_sync": (st, [vp, i64]),
        "psi_stream_wait": (st, [vp, i64]),
        "psi_arena_stats": (st, [vp, C.POINTER(psi_stats)]),
        "psi_kernel_launches": (C.c_uint64, []),
        "psi_arena_reset_stats": (st, [vp]),
        "psi_arena_set_timing": (st, [vp, i32]),
        "psi_arena_trace_begin": (st, [vp, sz]),
        "psi_arena_trace_get": (st, [vp, C.POINTER(psi_trace_record), sz, C.POINTER(sz)]),
        "psi_arena_fail_next_copy": (st, [vp]),
        "psi_debug_stall_next_gemm": (st, [C.c_uint64]),
        "psi_linear_paged": (st, [vp, vp, i64, i64, C.POINTER(psi_linear_weight), vp, vp,
                                  vp, i64, u32]),
        "psi_linear_rope_paged": (st, [vp, vp, i64, i64, C.POINTER(psi_linear_weight), vp,
                                       C.POINTER(psi_rope), vp, i64, u32]),
        "psi_rmsnorm": (st, [vp, i64, i64, i64, vp, C.c_float, vp, i64, vp]),
        "psi_ffn_paged": (st, [vp, vp, i64, C.POINTER(psi_ffn_weight), vp, vp, vp, vp, vp,
                               vp, u32]),
        "psi_ffn_paged_strided": (st, [vp, vp, i64, C.POINTER(psi_ffn_weight), vp, vp, vp, vp, vp,
                                       vp, i64, u32]),
        "psi_attn_partitioned": (st, [C.POINTER(psi_heads)] * 4 +
                                 [i32, i64, i64, i32, C.c_float, i32, vp, u32]),
        "psi_attn_partitioned_ws": (st, [C.POINTER(psi_heads)] * 4 +
                                    [i32, i64, i64, i32, C.c_float, i32, vp, sz, vp, u32]),
        "psi_attn_workspace_size": (st, [i32, C.POINTER(sz)]),
        "psi_ffn_resident_noalloc": (st, [vp, i64, C.POINTER(psi_ffn_weight), vp, vp, vp, vp,
                                          vp, u32]),
        "psi_journal_create": (st, [vp, vp, sz, sz, C.POINTER(vp)]),
        "psi_journal_destroy": (st, [vp]),
        "psi_journal_commit": (st, [vp, psi_key, vp, sz]),
        "psi_journal_reload": (st, [vp, psi_key, vp, sz]),
        "psi_journal_acquire": (st, [vp, psi_key]),
        "psi_journal_fence": (st, [vp, vp, sz]),
        "psi_journal_drop": (st, [vp, psi_key]),
        "psi_journal_host_view": (st, [vp, psi_key, i64, C.POINTER(vp), C.POINTER(sz)]),
        "psi_journal_get_stats": (st, [vp, C.POINTER(psi_journal_stats)]),
        "psi_journal_fail_next_copy": (st, [vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != PSI_OK:
        raise PsiError(status, load().psi_last_error().decode())


# ------------------------------------------------------------- wrappers --
def psi_version() -> str:
    return load().psi_version().decode()


def psi_status_string(s: int) -> str:
    return load().psi_status_string(s).decode()


def psi_last_error() -> str:
    return load().psi_last_error().decode()


def psi_plan_linear(rows: int, cols: int, page_bytes: int) -> int:
    out = C.c_int64()
    _check(load().psi_plan_linear(rows, cols, page_bytes, C.byref(out)))
    return out.value


def psi_plan_columns(cols: int, align: int, parts: int, part: int) -> tuple[int, int]:
    c0, c1 = C.c_int64(), C.c_int64()
    _check(load().psi_plan_columns(cols, align, parts, part, C.byref(c0), C.byref(c1)))
    return c0.value, c1.value


def psi_ffn_page_bytes(d: int, r: int, slice_: int) -> int:
    return load().psi_ffn_page_bytes(d, r, slice_)


def psi_ffn_pack(U: int, V: int, d: int, h: int, r: int, slice_: int, dst: int):
    _check(load().psi_ffn_pack(U, V, d, h, r, slice_, dst))


def psi_ffn_workspace(N: int, r: int, slice_: int):
    hb, ab = C.c_size_t(), C.c_size_t()
    _check(load().psi_ffn_workspace(N, r, slice_, C.byref(hb), C.byref(ab)))
    return hb.value, ab.value


def psi_arena_create(dev_base: int, dev_bytes: int, page_bytes: int,
                     compute_stream: int, copy_stream: int) -> int:
    out = C.c_void_p()
    _check(load().psi_arena_create(dev_base, dev_bytes, page_bytes, compute_stream,
                                   copy_stream, C.byref(out)))
    return out.value


def psi_arena_destroy(arena: int):
    _check(load().psi_arena_destroy(arena))


def psi_arena_slots(arena: int) -> int:
    return load().psi_arena_slots(arena)


def psi_page_stream(arena: int, host_src: int, nbytes: int, flags: int = 0) -> psi_page:
    pg = psi_page()
    _check(load().psi_page_stream(arena, host_src, nbytes, flags, C.byref(pg)))
    return pg


def psi_page_release(arena: int, page: psi_page):
    _check(load().psi_page_release(arena, page))


def psi_sync(arena: int, timeout_ms: int = 60000):
    _check(load().psi_sync(arena, timeout_ms))


def psi_stream_wait(stream: int, timeout_ms: int = 60000):
    _check(load().psi_stream_wait(stream, timeout_ms))


def psi_arena_stats(arena: int) -> dict:
    s = psi_stats()
    _check(load().psi_arena_stats(arena, C.byref(s)))
    return s.as_dict()


def psi_arena_reset_stats(arena: int):
    _check(load().psi_arena_reset_stats(arena))


def psi_arena_set_timing(arena: int, enable: bool):
    _check(load().psi_arena_set_timing(arena, 1 if enable else 0))


def psi_arena_trace_begin(arena: int, capacity: int):
    _check(load().psi_arena_trace_begin(arena, capacity))


def psi_arena_trace_get(arena: int) -> list:
    """The page timeline records held (ordered by start time) as dicts."""
    n = C.c_size_t(0)
    _check(load().psi_arena_trace_get(arena, None, 0, C.byref(n)))
    buf = (psi_trace_record * max(n.value, 1))()
    _check(load().psi_arena_trace_get(arena, buf, n.value, C.byref(n)))
    return [buf[i].as_dict() for i in range(n.value)]


def psi_arena_fail_next_copy(arena: int):
    _check(load().psi_arena_fail_next_copy(arena))


def psi_kernel_launches() -> int:
    """Kernels the library has launched in this process."""
    return load().psi_kernel_launches()


def psi_debug_stall_next_gemm(timeout_ns: int):
    _check(load().psi_debug_stall_next_gemm(timeout_ns))


def psi_linear_paged(arena: int, X: int, N: int, K: int, W: psi_linear_weight, bias: int,
                     residual: int | None, Y: int, ldy: int, flags: int = 0):
    _check(load().psi_linear_paged(arena, X, N, K, C.byref(W), bias, residual or None, Y,
                                   ldy, flags))


def psi_linear_rope_paged(arena: int, X: int, N: int, K: int, W: psi_linear_weight, bias: int,
                          rope: psi_rope, Y: int, ldy: int, flags: int = 0):
    _check(load().psi_linear_rope_paged(arena, X, N, K, C.byref(W), bias, C.byref(rope), Y,
                                        ldy, flags))


def psi_rmsnorm(X: int, ldx: int, N: int, d: int, gamma: int, eps: float, Y: int, ldy: int,
                stream: int):
    _check(load().psi_rmsnorm(X, ldx, N, d, gamma, eps, Y, ldy, stream))


def psi_ffn_paged(arena: int, X: int, N: int, W: psi_ffn_weight, a: int, b: int,
                  hidden_ws: int, acc_ws: int, residual: int | None, Y: int, flags: int = 0):
    _check(load().psi_ffn_paged(arena, X, N, C.byref(W), a, b, hidden_ws, acc_ws,
                                residual or None, Y, flags))


def psi_ffn_paged_strided(arena: int, X: int, N: int, W: psi_ffn_weight, a: int, b: int,
                          hidden_ws: int, acc_ws: int, residual: int | None, Y: int, ldy: int,
                          flags: int = 0):
    _check(load().psi_ffn_paged_strided(arena, X, N, C.byref(W), a, b, hidden_ws, acc_ws,
                                        residual or None, Y, ldy, flags))


def psi_attn_partitioned(Q: psi_heads, K: psi_heads, V: psi_heads, O: psi_heads, heads: int,
                         Nq: int, Nk: int, dh: int, scale: float, key_block: int, stream: int,
                         flags: int = 0):
    _check(load().psi_attn_partitioned(C.byref(Q), C.byref(K), C.byref(V), C.byref(O), heads,
                                       Nq, Nk, dh, scale, key_block, stream, flags))


def psi_attn_partitioned_ws(Q: psi_heads, K: psi_heads, V: psi_heads, O: psi_heads,
                            heads: int, Nq: int, Nk: int, dh: int, scale: float, key_block: int,
                            workspace: int | None, workspace_bytes: int, stream: int,
                            flags: int = 0):
    _check(load().psi_attn_partitioned_ws(C.byref(Q), C.byref(K), C.byref(V), C.byref(O), heads,
                                          Nq, Nk, dh, scale, key_block, workspace or None,
                                          workspace_bytes, stream, flags))


def psi_attn_workspace_size(key_block: int) -> int:
    n = C.c_size_t()
    _check(load().psi_attn_workspace_size(key_block, C.byref(n)))
    return n.value


def psi_ffn_resident_noalloc(X: int, N: int, W: psi_ffn_weight, a: int, b: int,
                             residual: int | None, Y: int, stream: int, flags: int = 0):
    """FFN with resident weights and the library's fixed workspace (for
    callers that cannot allocate device memory); see include/psi.h."""
    _check(load().psi_ffn_resident_noalloc(X, N, C.byref(W), a, b, residual or None, Y,
                                           stream, flags))


# ------------------------------------------------------------- journal ---
def psi_journal_create(arena: int, host: int, host_bytes: int, slot_bytes: int) -> int:
    out = C.c_void_p()
    _check(load().psi_journal_create(arena, host, host_bytes, slot_bytes, C.byref(out)))
    return out.value


def psi_journal_destroy(j: int):
    _check(load().psi_journal_destroy(j))


def _key(k) -> psi_key:
    return k if isinstance(k, psi_key) else psi_key(*k)


def psi_journal_commit(j: int, key, dev_src: int, nbytes: int):
    _check(load().psi_journal_commit(j, _key(key), dev_src, nbytes))


def psi_journal_reload(j: int, key, dev_dst: int, nbytes: int):
    _check(load().psi_journal_reload(j, _key(key), dev_dst, nbytes))


def psi_journal_acquire(j: int, key):
    _check(load().psi_journal_acquire(j, _key(key)))


def psi_journal_fence(j: int, dev_ptr: int, nbytes: int):
    _check(load().psi_journal_fence(j, dev_ptr, nbytes))


def psi_journal_drop(j: int, key):
    _check(load().psi_journal_drop(j, _key(key)))


def psi_journal_host_view(j: int, key, timeout_ms: int = 10000):
    """(host address, bytes) of a committed entry, after its copy finished."""
    p, n = C.c_void_p(), C.c_size_t()
    _check(load().psi_journal_host_view(j, _key(key), timeout_ms, C.byref(p), C.byref(n)))
    return p.value, n.value


def psi_journal_get_stats(j: int) -> dict:
    st = psi_journal_stats()
    _check(load().psi_journal_get_stats(j, C.byref(st)))
    return st.as_dict()


def psi_journal_fail_next_copy(j: int):
    _check(load().psi_journal_fail_next_copy(j))
