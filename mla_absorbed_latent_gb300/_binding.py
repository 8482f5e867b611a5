"""ctypes binding of libmla.so: the C ABI of include/mla.h, same names.

Argument marshalling only: torch tensors (device memory owned by the
caller) are passed as raw pointers, the stream defaults to torch's current
stream, and a negative status raises MLAError.  Every step of the decode
path runs in the library's CUDA kernels; there is no fallback of any kind:
if libmla.so is missing the import fails.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmla.so")

MLA_OK, MLA_ERR_INVALID, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA = 0, -1, -2, -3
MLA_ERR_BOUNDS, MLA_ERR_TIMEOUT, MLA_ERR_WORKSPACE = -4, -5, -6
FMT = {"bf16": 0, "int8": 1, "int4": 2, "int8_token": 3, "int4_sym": 4, "int4_pe4": 5}
D_C, D_R, D_NOPE, D_V, PAGE = 512, 64, 128, 128, 64
MLA_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024  # the fixed scratch of mla_decode_noalloc
MLA_KERNEL_CUDA_CORES, MLA_KERNEL_TCGEN05, MLA_KERNEL_MMA = 0, 1, 2  # mla_kernel_t


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.mla_status_string(status).decode()} ({status})")


class mla_cache_t(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("num_pages", ctypes.c_int), ("pages", ctypes.c_void_p)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first (python mla_absorbed_latent_gb300/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    cp = ctypes.POINTER(mla_cache_t)
    sigs = {
        "mla_cache_page_bytes": (sz, [i]),
        "mla_absorb_weights": (i, [vp, i, vp, vp, vp]),
        "mla_cache_append": (i, [cp, vp, vp, vp, i, vp, i, i, vp]),
        "mla_cache_project_append": (i, [cp, vp, i, vp, vp, f, f, vp, i, vp, i, i, vp, i, vp, sz, vp]),
        "mla_cache_project_workspace_bytes": (sz, [i, i, i, i]),
        "mla_decode_workspace_bytes": (sz, [i, i]),
        "mla_decode": (i, [vp, vp, vp, vp, i, cp, vp, i, vp, i, f, vp, sz, vp, vp]),
        "mla_decode_plan": (i, [i, i, vp, i, i, vp, sz, vp]),
        "mla_decode_plan_workers": (i, [i, i, vp, i, i, i, vp, sz, vp]),
        "mla_decode_max_workers": (i, [i, i]),
        "mla_decode_absorb_q": (i, [vp, vp, vp, i, i, vp, sz, vp]),
        "mla_decode_attend": (i, [i, cp, vp, i, vp, i, f, vp, sz, vp]),
        "mla_decode_combine": (i, [vp, i, i, vp, sz, vp, vp, vp]),
        "mla_decode_noalloc": (i, [vp, vp, vp, vp, i, cp, vp, i, vp, i, f, vp, vp]),
        "mla_decode_q": (i, [vp, vp, vp, vp, i, i, cp, vp, i, vp, i, f, vp, sz, vp, vp, vp]),
        "mla_decode_q_workspace_bytes": (sz, [i, i, i]),
        "mla_prefill": (i, [vp, vp, vp, i, i, cp, vp, i, vp, i, f, vp, sz, vp, vp]),
        "mla_prefill_workspace_bytes": (sz, [i, i, i]),
        "mla_output_projection": (i, [vp, vp, i, i, i, vp, vp, sz, vp]),
        "mla_output_projection_workspace_bytes": (sz, [i, i, i]),
        "mla_get_device_status": (i, [vp, ctypes.POINTER(ctypes.c_int)]),
        "mla_wait_selftest": (i, [vp]),
        "mla_decode_kernel_kind": (i, [i]),
        "mla_decode_select_kernel": (i, [i, i]),
        "mla_status_string": (ctypes.c_char_p, [i]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str) -> None:
    if status != MLA_OK:
        raise MLAError(status, where)


def cache_struct(fmt: str | int, num_pages: int, pages) -> mla_cache_t:
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    return mla_cache_t(f, int(num_pages), _ptr(pages))


def mla_cache_page_bytes(fmt: str | int) -> int:
    return int(_lib.mla_cache_page_bytes(FMT[fmt] if isinstance(fmt, str) else int(fmt)))


def mla_absorb_weights(wkv_b, H: int, W_UK, W_UV, stream=None) -> None:
    _check(_lib.mla_absorb_weights(_ptr(wkv_b), H, _ptr(W_UK), _ptr(W_UV), _stream(stream)), "mla_absorb_weights")


def mla_cache_append(cache: mla_cache_t, c_kv, k_pe, page_table, max_pages: int, pos, B: int, T: int,
                     stream=None) -> None:
    _check(_lib.mla_cache_append(ctypes.byref(cache), _ptr(c_kv), _ptr(k_pe), _ptr(page_table), max_pages,
                                 _ptr(pos), B, T, _stream(stream)), "mla_cache_append")


def mla_cache_project_workspace_bytes(B: int, T: int, hidden: int, k_splits: int = 0) -> int:
    return int(_lib.mla_cache_project_workspace_bytes(B, T, hidden, k_splits))


def mla_cache_project_append(cache: mla_cache_t, x, hidden: int, wkv_a, kv_norm_w, eps: float, rope_theta: float,
                             page_table, max_pages: int, pos, B: int, T: int, latent_out=None, k_splits: int = 0,
                             workspace=None, workspace_bytes: int = 0, stream=None) -> None:
    _check(_lib.mla_cache_project_append(ctypes.byref(cache), _ptr(x), hidden, _ptr(wkv_a), _ptr(kv_norm_w), eps,
                                         rope_theta, _ptr(page_table), max_pages, _ptr(pos), B, T, _ptr(latent_out),
                                         k_splits, _ptr(workspace), workspace_bytes, _stream(stream)),
           "mla_cache_project_append")


def mla_decode_workspace_bytes(B: int, H: int) -> int:
    return int(_lib.mla_decode_workspace_bytes(B, H))


def mla_decode(q_nope, q_pe, W_UK, W_UV, H: int, cache: mla_cache_t, page_table, max_pages: int, seqlens,
               B: int, scale: float, workspace, workspace_bytes: int, out, stream=None) -> None:
    _check(_lib.mla_decode(_ptr(q_nope), _ptr(q_pe), _ptr(W_UK), _ptr(W_UV), H, ctypes.byref(cache),
                           _ptr(page_table), max_pages, _ptr(seqlens), B, scale, _ptr(workspace),
                           workspace_bytes, _ptr(out), _stream(stream)), "mla_decode")


def mla_decode_q_workspace_bytes(B: int, H: int, T: int) -> int:
    return int(_lib.mla_decode_q_workspace_bytes(B, H, T))


def mla_decode_q(q_nope, q_pe, W_UK, W_UV, H: int, T: int, cache: mla_cache_t, page_table, max_pages: int, seqlens,
                 B: int, scale: float, workspace, workspace_bytes: int, out, o_lat_out=None, stream=None) -> None:
    """T causal query tokens per row (the last T cached tokens of each row)."""
    _check(_lib.mla_decode_q(_ptr(q_nope), _ptr(q_pe), _ptr(W_UK), _ptr(W_UV), H, T, ctypes.byref(cache),
                             _ptr(page_table), max_pages, _ptr(seqlens), B, scale, _ptr(workspace), workspace_bytes,
                             _ptr(out), _ptr(o_lat_out), _stream(stream)), "mla_decode_q")


def mla_prefill_workspace_bytes(B: int, H: int, max_pages: int) -> int:
    return int(_lib.mla_prefill_workspace_bytes(B, H, max_pages))


def mla_prefill(q_nope, q_pe, wkv_b, H: int, T: int, cache: mla_cache_t, page_table, max_pages: int, seqlens, B: int,
                scale: float, workspace, workspace_bytes: int, out, stream=None) -> None:
    """The unabsorbed causal prefill (expanded keys and values, standard attention)."""
    _check(_lib.mla_prefill(_ptr(q_nope), _ptr(q_pe), _ptr(wkv_b), H, T, ctypes.byref(cache), _ptr(page_table),
                            max_pages, _ptr(seqlens), B, scale, _ptr(workspace), workspace_bytes, _ptr(out),
                            _stream(stream)), "mla_prefill")


def mla_output_projection_workspace_bytes(R: int, H: int, hidden: int) -> int:
    return int(_lib.mla_output_projection_workspace_bytes(R, H, hidden))


def mla_output_projection(o, W_O, R: int, H: int, hidden: int, y, workspace=None, workspace_bytes: int = 0,
                          stream=None) -> None:
    """y [R][hidden] = o [R][H*128] W_O^T (the step after the value up-projection)."""
    _check(_lib.mla_output_projection(_ptr(o), _ptr(W_O), R, H, hidden, _ptr(y), _ptr(workspace), workspace_bytes,
                                      _stream(stream)), "mla_output_projection")


def mla_decode_plan(H: int, fmt: str | int, seqlens, B: int, max_pages: int, workspace, workspace_bytes: int,
                    stream=None) -> None:
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    _check(_lib.mla_decode_plan(H, f, _ptr(seqlens), B, max_pages, _ptr(workspace), workspace_bytes,
                                _stream(stream)), "mla_decode_plan")


def mla_decode_plan_workers(H: int, fmt: str | int, seqlens, B: int, max_pages: int, workers: int, workspace,
                            workspace_bytes: int, stream=None) -> None:
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    _check(_lib.mla_decode_plan_workers(H, f, _ptr(seqlens), B, max_pages, workers, _ptr(workspace),
                                        workspace_bytes, _stream(stream)), "mla_decode_plan_workers")


def mla_decode_max_workers(H: int, fmt: str | int = "bf16") -> int:
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    n = int(_lib.mla_decode_max_workers(H, f))
    _check(min(n, 0), "mla_decode_max_workers")
    return n


def mla_decode_absorb_q(q_nope, q_pe, W_UK, H: int, B: int, workspace, workspace_bytes: int, stream=None) -> None:
    _check(_lib.mla_decode_absorb_q(_ptr(q_nope), _ptr(q_pe), _ptr(W_UK), H, B, _ptr(workspace),
                                    workspace_bytes, _stream(stream)), "mla_decode_absorb_q")


def mla_decode_attend(H: int, cache: mla_cache_t, page_table, max_pages: int, seqlens, B: int, scale: float,
                      workspace, workspace_bytes: int, stream=None) -> None:
    _check(_lib.mla_decode_attend(H, ctypes.byref(cache), _ptr(page_table), max_pages, _ptr(seqlens), B, scale,
                                  _ptr(workspace), workspace_bytes, _stream(stream)), "mla_decode_attend")


def mla_decode_combine(W_UV, H: int, B: int, workspace, workspace_bytes: int, out, o_lat_out=None,
                       stream=None) -> None:
    _check(_lib.mla_decode_combine(_ptr(W_UV), H, B, _ptr(workspace), workspace_bytes, _ptr(out),
                                   _ptr(o_lat_out), _stream(stream)), "mla_decode_combine")


def mla_get_device_status(stream=None) -> tuple[int, int]:
    """(status, detail) of the first device-detected error since the last call; clears it."""
    info = ctypes.c_int(0)
    st = _lib.mla_get_device_status(_stream(stream), ctypes.byref(info))
    return int(st), int(info.value)


def mla_wait_selftest(stream=None) -> None:
    """Enqueue the bounded-wait self-test (about 2 s on the device); read its
    outcome with mla_get_device_status."""
    _check(_lib.mla_wait_selftest(_stream(stream)), "mla_wait_selftest")


def mla_decode_kernel_kind(H: int) -> int:
    return int(_lib.mla_decode_kernel_kind(H))


def mla_decode_select_kernel(H: int, kind: int) -> None:
    """Process-wide choice of the attend kernel for H heads (see include/mla.h)."""
    _check(_lib.mla_decode_select_kernel(H, kind), "mla_decode_select_kernel")


def mla_status_string(status: int) -> str:
    return _lib.mla_status_string(status).decode()


def mla_decode_noalloc(q_nope, q_pe, W_UK, W_UV, H: int, cache: mla_cache_t, page_table, max_pages: int, seqlens,
                       B: int, scale: float, out, stream=None) -> None:
    """mla_decode with the library's fixed device scratch instead of a workspace
    (for hosts that cannot allocate; see include/mla.h)."""
    _check(_lib.mla_decode_noalloc(_ptr(q_nope), _ptr(q_pe), _ptr(W_UK), _ptr(W_UV), H, ctypes.byref(cache),
                                   _ptr(page_table), max_pages, _ptr(seqlens), B, scale, _ptr(out), _stream(stream)),
           "mla_decode_noalloc")


def raw_library() -> ctypes.CDLL:
    """The loaded ctypes library (for callers that marshal arguments themselves)."""
    return _lib
