"""Thin Python binding of the libnk C ABI (``include/nk.h``).

Argument marshalling only: every step of the hot path runs in libnk's CUDA
kernels.  Functions named ``nk_*`` mirror the C entry points one to one and
take raw integers for device pointers and streams; ``Pool`` is a convenience
wrapper that allocates the planes as torch tensors (device memory), keeps them
alive and passes ``torch.cuda.current_stream()``.

There is no CPU fallback: ``load()`` raises when ``libnk.so`` has not been
built, and every call raises ``NkError`` on a non-zero status.
"""

from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libnk.so")

NK_OK = 0
ERRORS = {-1: "NK_ERR_INVALID_ARG", -2: "NK_ERR_SHAPE", -3: "NK_ERR_RANGE",
          -4: "NK_ERR_UNSUPPORTED", -5: "NK_ERR_ALIGN", -6: "NK_ERR_CUDA", -7: "NK_ERR_WORKSPACE"}
STATUS_PAGE_RANGE, STATUS_FRONTIER, STATUS_TIMEOUT = 1, 2, 4
PROFILES = {"bf16": 0, "int8_g64": 1, "fp8_row": 2, "nvfp4_g16": 3, "k8v4": 4}
POOL_CHECK_BOUNDS = 1

SYMBOLS = ["nk_version", "nk_last_error", "nk_pool_plane_bytes", "nk_pool_capacity_bounds",
           "nk_pool_mtp_pages", "nk_pages_needed",
           "nk_pool_create", "nk_pool_destroy", "nk_paged_kv_append", "nk_decode_workspace_bytes",
           "nk_paged_decode_attention", "nk_paged_append_decode_attention",
           "nk_paged_decode_attention_noalloc",
           "nk_prefill_workspace_bytes", "nk_paged_prefill_attention",
           "nk_page_copy_columns", "nk_status_read", "nk_host_page_bytes", "nk_page_runs",
           "nk_pages_to_host", "nk_pages_from_host", "nk_selftest_bounded_wait"]


class NkError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class PoolDesc(C.Structure):
    _fields_ = [("profile", C.c_int32), ("num_layers", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("max_context", C.c_int32),
                ("max_concurrency", C.c_int32), ("order", C.c_int32), ("flags", C.c_int32)]


_lib = None
_P, _I, _F, _S = C.c_void_p, C.c_int32, C.c_float, C.c_size_t


def load(path: str | None = None) -> C.CDLL:
    """Loads libnk.so (raises RuntimeError when it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is not built; run paged_kv_cache_append_gb300.build.build()")
    lib = C.CDLL(p)
    sig = {
        "nk_version": (C.c_int, []),
        "nk_last_error": (C.c_char_p, []),
        "nk_pool_plane_bytes": (C.c_int, [C.POINTER(PoolDesc), _I, C.POINTER(_I), C.POINTER(_S), C.POINTER(_S)]),
        "nk_pool_capacity_bounds": (C.c_int, [C.POINTER(PoolDesc), C.POINTER(_I), C.POINTER(_I)]),
        "nk_pool_create": (C.c_int, [C.POINTER(PoolDesc), _I, C.POINTER(_P), C.POINTER(_P)]),
        "nk_pool_destroy": (C.c_int, [_P]),
        "nk_paged_kv_append": (C.c_int, [_P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _P]),
        "nk_pool_mtp_pages": (C.c_int, [_I, _I, _I, C.POINTER(_I)]),
        "nk_pages_needed": (C.c_int, [_I, _I, C.POINTER(_I)]),
        "nk_host_page_bytes": (C.c_int, [_P, C.POINTER(_S)]),
        "nk_page_runs": (C.c_int, [_P, _I, _P, _P, C.POINTER(_I)]),
        "nk_pages_to_host": (C.c_int, [_P, _P, _I, _P, _P]),
        "nk_pages_from_host": (C.c_int, [_P, _P, _I, _P, _P]),
        "nk_decode_workspace_bytes": (C.c_int, [_P, _I, _I, _I, C.POINTER(_S)]),
        "nk_paged_decode_attention": (C.c_int, [_P, _I, _P, _I, _P, _P, _P, _I, _I, _F, _P, _P, _P, _S, _P]),
        "nk_paged_append_decode_attention": (C.c_int, [_P, _I, _P, _I, _P, _P, _P, _P, _P, _I, _I, _F, _P, _P, _P,
                                                       _S, _P]),
        "nk_paged_decode_attention_noalloc": (C.c_int, [_P, _I, _P, _I, _P, _P, _P, _I, _I, _F, _P, _P, _P]),
        "nk_prefill_workspace_bytes": (C.c_int, [_P, _I, _I, _I, C.POINTER(_S)]),
        "nk_paged_prefill_attention": (C.c_int, [_P, _I, _P, _I, _P, _P, _P, _P, _I, _I, _F, _P, _P, _P, _S, _P]),
        "nk_page_copy_columns": (C.c_int, [_P, _I, _I, _I, _P]),
        "nk_status_read": (C.c_int, [C.POINTER(_I), _I, _P]),
        "nk_selftest_bounded_wait": (C.c_int, [_I, _P, _P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != NK_OK:
        raise NkError(rc, load().nk_last_error().decode())


ORDERS = {"page_major": 0, "head_major": 1}


def make_desc(profile, num_layers, num_kv_heads, head_dim, max_context, max_concurrency,
              flags: int = 0, order: str = "page_major") -> PoolDesc:
    prof = PROFILES[profile] if isinstance(profile, str) else int(profile)
    return PoolDesc(prof, num_layers, num_kv_heads, head_dim, max_context, max_concurrency,
                    ORDERS[order], flags)


# ----------------------------------------------------------- C-named wrappers

def nk_version() -> int:
    return load().nk_version()


def nk_pool_plane_bytes(desc: PoolDesc, M: int):
    n = _I()
    b = (_S * 4)()
    rb = (_S * 4)()
    _check(load().nk_pool_plane_bytes(C.byref(desc), M, C.byref(n), b, rb))
    return n.value, list(b)[:n.value], list(rb)[:n.value]


def nk_pool_capacity_bounds(desc: PoolDesc):
    lo, hi = _I(), _I()
    _check(load().nk_pool_capacity_bounds(C.byref(desc), C.byref(lo), C.byref(hi)))
    return lo.value, hi.value


def nk_pool_create(desc: PoolDesc, M: int, plane_ptrs) -> int:
    arr = (_P * len(plane_ptrs))(*plane_ptrs)
    out = _P()
    _check(load().nk_pool_create(C.byref(desc), M, arr, C.byref(out)))
    return out.value


def nk_pool_destroy(pool: int) -> None:
    _check(load().nk_pool_destroy(pool))


def nk_paged_kv_append(pool, layer, block_tables, table_rows, write_pos, counts, k, v, B, T, stream):
    _check(load().nk_paged_kv_append(pool, layer, block_tables, table_rows, write_pos, counts,
                                     k, v, B, T, stream))


def nk_pool_mtp_pages(M, C_rows, draft_window) -> int:
    n = _I()
    _check(load().nk_pool_mtp_pages(M, C_rows, draft_window, C.byref(n)))
    return n.value


def nk_pages_needed(committed_frontier, provisional_frontier) -> int:
    n = _I()
    _check(load().nk_pages_needed(committed_frontier, provisional_frontier, C.byref(n)))
    return n.value


def nk_page_runs(page_ids):
    """Runs of consecutive physical ids: list of (first logical page, length)."""
    import numpy as np
    ids = np.ascontiguousarray(page_ids, dtype=np.int32)
    n = ids.size
    first = np.zeros(max(n, 1), np.int32)
    ln = np.zeros(max(n, 1), np.int32)
    nr = _I()
    _check(load().nk_page_runs(ids.ctypes.data, n, first.ctypes.data, ln.ctypes.data, C.byref(nr)))
    return [(int(first[r]), int(ln[r])) for r in range(nr.value)]


def nk_decode_workspace_bytes(pool, B, T, Hq) -> int:
    n = _S()
    _check(load().nk_decode_workspace_bytes(pool, B, T, Hq, C.byref(n)))
    return n.value


def nk_paged_decode_attention(q, Hq, pool, layer, block_tables, table_rows, frontiers, B, T, scale,
                              out, lse, workspace, workspace_bytes, stream):
    _check(load().nk_paged_decode_attention(q, Hq, pool, layer, block_tables, table_rows, frontiers,
                                            B, T, scale, out, lse, workspace, workspace_bytes, stream))


def nk_paged_append_decode_attention(q, Hq, pool, layer, block_tables, table_rows, frontiers, k, v, B,
                                     T, scale, out, lse, workspace, workspace_bytes, stream):
    _check(load().nk_paged_append_decode_attention(q, Hq, pool, layer, block_tables, table_rows,
                                                   frontiers, k, v, B, T, scale, out, lse, workspace,
                                                   workspace_bytes, stream))


def nk_paged_decode_attention_noalloc(q, Hq, pool, layer, block_tables, table_rows, frontiers, B, T,
                                      scale, out, lse, stream):
    _check(load().nk_paged_decode_attention_noalloc(q, Hq, pool, layer, block_tables, table_rows,
                                                    frontiers, B, T, scale, out, lse, stream))


def nk_prefill_workspace_bytes(pool, B, Tc, Hq) -> int:
    n = _S()
    _check(load().nk_prefill_workspace_bytes(pool, B, Tc, Hq, C.byref(n)))
    return n.value


def nk_paged_prefill_attention(q, Hq, pool, layer, block_tables, table_rows, prefix_len, chunk_len,
                               B, Tc, scale, out, lse, workspace, workspace_bytes, stream):
    _check(load().nk_paged_prefill_attention(q, Hq, pool, layer, block_tables, table_rows, prefix_len,
                                             chunk_len, B, Tc, scale, out, lse, workspace,
                                             workspace_bytes, stream))


def nk_page_copy_columns(pool, src, dst, ncols, stream):
    _check(load().nk_page_copy_columns(pool, src, dst, ncols, stream))


def nk_status_read(clear: bool = True, stream=None) -> int:
    s = _I()
    _check(load().nk_status_read(C.byref(s), int(clear), stream))
    return s.value


def nk_selftest_bounded_wait(limit_us: int, waited_ns_ptr=None, stream=None) -> None:
    _check(load().nk_selftest_bounded_wait(int(limit_us), waited_ns_ptr, stream))


# ------------------------------------------------------------ torch wrapper

def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class Pool:
    """A typed growing KV pool whose planes are torch uint8 device tensors.

    ``planes[layer][i]`` follows nk.h's plane order [K code, V code, K scale,
    V scale]; ``tables`` etc. are int32 device tensors owned by the caller.
    """

    def __init__(self, profile: str, num_layers: int, num_kv_heads: int, head_dim: int,
                 max_context: int, max_concurrency: int, M: int, device="cuda",
                 check_bounds: bool = False, order: str = "page_major"):
        import torch
        self.profile, self.num_layers, self.H, self.D = profile, num_layers, num_kv_heads, head_dim
        self.S, self.C, self.M = max_context, max_concurrency, M
        self.L = -(-max_context // 64)
        self.order = order
        self.desc = make_desc(profile, num_layers, num_kv_heads, head_dim, max_context,
                              max_concurrency, POOL_CHECK_BOUNDS if check_bounds else 0, order)
        self.n_planes, self.plane_bytes, self.row_bytes = nk_pool_plane_bytes(self.desc, M)
        self.planes = [[torch.zeros(nb, dtype=torch.uint8, device=device) for nb in self.plane_bytes]
                       for _ in range(num_layers)]
        ptrs = [p.data_ptr() for layer in self.planes for p in layer]
        self.handle = nk_pool_create(self.desc, M, ptrs)
        self._ws = None

    def close(self) -> None:
        if self.handle:
            nk_pool_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def kv_bytes_per_token_head(self) -> int:
        return int(sum(self.row_bytes))

    def append(self, layer, tables, table_rows, write_pos, k, v, counts=None, stream=None):
        B, T = k.shape[0], k.shape[1]
        nk_paged_kv_append(self.handle, layer, _ptr(tables), _ptr(table_rows), _ptr(write_pos),
                           _ptr(counts), _ptr(k), _ptr(v), B, T, _stream(stream))

    def workspace(self, B, T, Hq):
        import torch
        n = nk_decode_workspace_bytes(self.handle, B, T, Hq)
        if self._ws is None or self._ws.numel() < n:   # zero-filled once (split counters)
            self._ws = torch.zeros(max(n, 16), dtype=torch.uint8, device=self.planes[0][0].device)
        return self._ws

    def decode(self, layer, q, tables, table_rows, frontiers, scale, out=None, lse=None,
               workspace=None, stream=None):
        import torch
        B, T, Hq, D = q.shape
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, T, Hq), dtype=torch.float32, device=q.device)
        ws = workspace if workspace is not None else self.workspace(B, T, Hq)
        nk_paged_decode_attention(_ptr(q), Hq, self.handle, layer, _ptr(tables), _ptr(table_rows),
                                  _ptr(frontiers), B, T, float(scale), _ptr(out), _ptr(lse),
                                  _ptr(ws), ws.numel(), _stream(stream))
        return out, lse

    def append_decode(self, layer, q, k, v, tables, table_rows, frontiers, scale, out=None, lse=None,
                      workspace=None, stream=None):
        """Appends the T new tokens k, v [B, T, H, D] of every row at
        frontiers - T .. frontiers - 1, then attends (one launch)."""
        import torch
        B, T, Hq, D = q.shape
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, T, Hq), dtype=torch.float32, device=q.device)
        ws = workspace if workspace is not None else self.workspace(B, T, Hq)
        nk_paged_append_decode_attention(_ptr(q), Hq, self.handle, layer, _ptr(tables), _ptr(table_rows),
                                         _ptr(frontiers), _ptr(k), _ptr(v), B, T, float(scale), _ptr(out),
                                         _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
        return out, lse

    def host_page_bytes(self) -> int:
        n = _S()
        _check(load().nk_host_page_bytes(self.handle, C.byref(n)))
        return n.value

    def pages_to_host(self, page_ids, host, stream=None):
        """Packs pages page_ids (logical order) into the uint8 host tensor
        `host` [n, host_page_bytes] (asynchronous when it is pinned)."""
        import numpy as np
        ids = np.ascontiguousarray(page_ids, dtype=np.int32)
        _check(load().nk_pages_to_host(self.handle, ids.ctypes.data, ids.size, host.data_ptr(),
                                       _stream(stream)))
        return host

    def pages_from_host(self, page_ids, host, stream=None):
        import numpy as np
        ids = np.ascontiguousarray(page_ids, dtype=np.int32)
        _check(load().nk_pages_from_host(self.handle, ids.ctypes.data, ids.size, host.data_ptr(),
                                         _stream(stream)))

    def prefill(self, layer, q, tables, table_rows, prefix_len, chunk_len, scale, out=None,
                lse=None, workspace=None, stream=None):
        import torch
        B, Tc, Hq, D = q.shape
        if out is None:
            out = torch.zeros_like(q)
        if lse is None:
            lse = torch.full((B, Tc, Hq), float("-inf"), dtype=torch.float32, device=q.device)
        n = nk_prefill_workspace_bytes(self.handle, B, Tc, Hq)
        ws = workspace
        if ws is None and n:   # split partials and counters, zero-filled once, kept for reuse
            if getattr(self, "_pws", None) is None or self._pws.numel() < n:
                self._pws = torch.zeros(n, dtype=torch.uint8, device=q.device)
            ws = self._pws
        nk_paged_prefill_attention(_ptr(q), Hq, self.handle, layer, _ptr(tables), _ptr(table_rows),
                                   _ptr(prefix_len), _ptr(chunk_len), B, Tc, float(scale), _ptr(out),
                                   _ptr(lse), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream))
        return out, lse

    def copy_columns(self, src, dst, ncols, stream=None):
        nk_page_copy_columns(self.handle, src, dst, ncols, _stream(stream))
