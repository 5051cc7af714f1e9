"""Thin ctypes binding over libmla.so (include/mla.h), with the same names as the C ABI.

Argument marshalling only: every step of the decode path runs in the
library's CUDA kernels.  Tensors are torch tensors on the CUDA device (torch
provides device memory and streams); their data pointers are passed as plain
device pointers.  There is no CPU fallback: if the library is missing or
cannot be loaded, :func:`load` raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libmla.so")

MLA_OK = 0
MLA_ERR_MISSING_FIELD = 1
MLA_ERR_INVALID_ARG = 2
MLA_ERR_UNSUPPORTED = 3
MLA_ERR_WORKSPACE = 4
MLA_ERR_CUDA = 5
MLA_ERR_DEVICE_CHECK = 6

MLA_CACHE_BF16 = 1
MLA_CACHE_FP8_E4M3 = 2
MLA_CACHE_FP8_E4M3_BLOCK = 3

MLA_CHECK_CTX_LEN = 0x1
MLA_CHECK_PAGE_ID = 0x2
MLA_CHECK_APPEND_INDEX = 0x4
MLA_CHECK_TIMEOUT = 0x8

MLA_OPT_SPLITS = 1
MLA_OPT_PROFILE = 2
MLA_OPT_TEST_STALL = 3
MLA_OPT_FP8_MMA = 4
MLA_OPT_SMALL_HEADS = 5

MLA_FIXED_SCRATCH_BYTES = 32 << 20     # include/mla.h: scratch of mla_decode_fixed_scratch

EXPORTED = [
    "mla_create", "mla_destroy", "mla_kv_append", "mla_kv_project_append", "mla_project",
    "mla_rmsnorm", "mla_expand_kv", "mla_decode_naive_workspace_size", "mla_decode_naive",
    "mla_prefill_workspace_size", "mla_prefill",
    "mla_decode_workspace_size", "mla_decode",
    "mla_decode_fixed_scratch",
    "mla_get_status", "mla_set_option", "mla_profile_read", "mla_profile_kernel_name", "mla_profile_last_name",
    "mla_last_error", "mla_status_string",
]


class MlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status
        self.message = message


class MlaConfig(ctypes.Structure):
    _fields_ = [
        ("d_c", ctypes.c_int32), ("d_rope", ctypes.c_int32), ("n_h", ctypes.c_int32),
        ("d_nope", ctypes.c_int32), ("d_v", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("cache_dtype", ctypes.c_int32), ("max_position", ctypes.c_int32),
        ("rope_base", ctypes.c_float), ("softmax_scale", ctypes.c_float), ("fp8_scale", ctypes.c_float),
    ]


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmla.so (built by ``python -m mla_absorbed_latent_decode_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libmla.so not found at {p}; build it with "
                           "`python -m mla_absorbed_latent_decode_gb300.build`")
    lib = ctypes.CDLL(p)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.mla_create.argtypes = [ctypes.POINTER(MlaConfig), vp, vp, vp, ctypes.POINTER(vp)]
    lib.mla_destroy.argtypes = [vp]
    lib.mla_kv_append.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, vp, i32, vp]
    lib.mla_kv_project_append.argtypes = [vp, vp, i32, vp, vp, vp, i32, vp, i32, i32, vp, i32, vp]
    lib.mla_project.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp]
    lib.mla_rmsnorm.argtypes = [vp, vp, i32, i32, i32, vp, ctypes.c_float, vp, i32, vp]
    lib.mla_expand_kv.argtypes = [vp, vp, i32, vp, vp]
    lib.mla_decode_naive_workspace_size.argtypes = [vp, i32, i32, ctypes.POINTER(sz)]
    lib.mla_decode_naive.argtypes = [vp, vp, vp, i32, i32, vp, i32, vp, i32, vp, sz, vp, vp]
    lib.mla_prefill_workspace_size.argtypes = [vp, i32, i32, ctypes.POINTER(sz)]
    lib.mla_prefill.argtypes = [vp, vp, vp, vp, i32, i32, vp, i32, i32, vp, i32, vp, i32, vp, sz, vp, vp]
    lib.mla_decode_workspace_size.argtypes = [vp, i32, i32, ctypes.POINTER(sz)]
    lib.mla_decode.argtypes = [vp, vp, vp, i32, i32, vp, i32, vp, i32, vp, sz, vp, vp]
    lib.mla_decode_fixed_scratch.argtypes = [vp, vp, vp, i32, i32, vp, i32, vp, i32, vp, vp]
    lib.mla_get_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.mla_set_option.argtypes = [vp, i32, i64]
    lib.mla_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float), i32, ctypes.POINTER(i32)]
    lib.mla_profile_kernel_name.argtypes = [i32]
    lib.mla_profile_kernel_name.restype = ctypes.c_char_p
    lib.mla_profile_last_name.argtypes = [vp, i32]
    lib.mla_profile_last_name.restype = ctypes.c_char_p
    lib.mla_last_error.argtypes = []
    lib.mla_last_error.restype = ctypes.c_char_p
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_status_string.restype = ctypes.c_char_p
    for name in ("mla_create", "mla_destroy", "mla_kv_append", "mla_decode_workspace_size", "mla_decode",
                 "mla_decode_fixed_scratch",
                 "mla_get_status", "mla_set_option", "mla_profile_read"):
        getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _status_name(s: int) -> str:
    names = {0: "MLA_OK", 1: "MLA_ERR_MISSING_FIELD", 2: "MLA_ERR_INVALID_ARG", 3: "MLA_ERR_UNSUPPORTED",
             4: "MLA_ERR_WORKSPACE", 5: "MLA_ERR_CUDA", 6: "MLA_ERR_DEVICE_CHECK"}
    return names.get(s, f"status {s}")


def _check(status: int) -> None:
    if status != MLA_OK:
        raise MlaError(status, load().mla_last_error().decode())


def _ptr(t) -> int:
    """Device pointer of a tensor (None -> 0)."""
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


def make_config(n_h: int, cache_dtype: int = MLA_CACHE_BF16, max_position: int = 65536, d_c: int = 512,
                d_rope: int = 64, d_nope: int = 128, d_v: int = 128, page_size: int = 64,
                rope_base: float = 10000.0, softmax_scale: float = 0.0, fp8_scale: float = 0.0) -> MlaConfig:
    return MlaConfig(d_c, d_rope, n_h, d_nope, d_v, page_size, cache_dtype, max_position, rope_base,
                     softmax_scale, fp8_scale)


class Mla:
    """An ``mla_handle_t``.  Methods mirror the C calls and raise :class:`MlaError` on failure."""

    def __init__(self, config: MlaConfig, w_uk, w_uv, stream=None):
        lib = load()
        self._lib = lib
        self.config = config
        h = ctypes.c_void_p()
        _check(lib.mla_create(ctypes.byref(config), _ptr(w_uk), _ptr(w_uv), _stream(stream), ctypes.byref(h)))
        self._h = h

    def close(self) -> None:
        if getattr(self, "_h", None) and self._h.value:
            self._lib.mla_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def kv_append(self, rows, seq, pos, block_table, cache, num_pages: int, stream=None) -> None:
        n = int(seq.shape[0])
        bt_rows, bt_stride = int(block_table.shape[0]), int(block_table.shape[1])
        _check(self._lib.mla_kv_append(self._h, _ptr(rows), _ptr(seq), _ptr(pos), n, _ptr(block_table), bt_rows,
                                       bt_stride, _ptr(cache), int(num_pages), _stream(stream)))

    def kv_project_append(self, x, w_dkv, seq, pos, block_table, cache, num_pages: int, stream=None) -> None:
        n, hidden = int(x.shape[0]), int(x.shape[1])
        bt_rows, bt_stride = int(block_table.shape[0]), int(block_table.shape[1])
        _check(self._lib.mla_kv_project_append(self._h, _ptr(x), hidden, _ptr(w_dkv), _ptr(seq), _ptr(pos), n,
                                               _ptr(block_table), bt_rows, bt_stride, _ptr(cache), int(num_pages),
                                               _stream(stream)))

    def project(self, x, w, y, stream=None) -> None:
        m, k, n_out = int(x.shape[0]), int(x.shape[1]), int(w.shape[0])
        _check(self._lib.mla_project(self._h, _ptr(x), m, k, _ptr(w), n_out, _ptr(y), _stream(stream)))

    def rmsnorm(self, x, n: int, w, eps: float, y, stream=None) -> None:
        """RMSNorm of the first n values of every row of the 2-D tensor x into y (may be x)."""
        m, ld_x, ld_y = int(x.shape[0]), int(x.stride(0)), int(y.stride(0))
        _check(self._lib.mla_rmsnorm(self._h, _ptr(x), m, int(n), ld_x, _ptr(w), float(eps), _ptr(y), ld_y,
                                     _stream(stream)))

    def expand_kv(self, cache, num_pages: int, kvx, stream=None) -> None:
        _check(self._lib.mla_expand_kv(self._h, _ptr(cache), int(num_pages), _ptr(kvx), _stream(stream)))

    def decode_naive_workspace_size(self, batch: int, max_ctx: int) -> int:
        out = ctypes.c_size_t()
        _check(self._lib.mla_decode_naive_workspace_size(self._h, int(batch), int(max_ctx), ctypes.byref(out)))
        return int(out.value)

    def decode_naive(self, q, ctx_len, max_ctx: int, block_table, kvx, num_pages: int, workspace, out,
                     stream=None) -> None:
        batch = int(ctx_len.shape[0])
        ws_bytes = int(workspace.numel() * workspace.element_size())
        _check(self._lib.mla_decode_naive(self._h, _ptr(q), _ptr(ctx_len), batch, int(max_ctx), _ptr(block_table),
                                          int(block_table.shape[1]), _ptr(kvx), int(num_pages), _ptr(workspace),
                                          ws_bytes, _ptr(out), _stream(stream)))

    def prefill_workspace_size(self, batch: int, max_ctx: int) -> int:
        out = ctypes.c_size_t()
        _check(self._lib.mla_prefill_workspace_size(self._h, int(batch), int(max_ctx), ctypes.byref(out)))
        return int(out.value)

    def prefill(self, q, q_start, q_len, max_q: int, ctx_len, max_ctx: int, block_table, cache, num_pages: int,
                workspace, out, stream=None) -> None:
        batch, total_q = int(ctx_len.shape[0]), int(q.shape[0])
        ws_bytes = int(workspace.numel() * workspace.element_size())
        _check(self._lib.mla_prefill(self._h, _ptr(q), _ptr(q_start), _ptr(q_len), total_q, int(max_q), _ptr(ctx_len),
                                     batch, int(max_ctx), _ptr(block_table), int(block_table.shape[1]), _ptr(cache),
                                     int(num_pages), _ptr(workspace), ws_bytes, _ptr(out), _stream(stream)))

    def decode_workspace_size(self, batch: int, max_ctx: int) -> int:
        out = ctypes.c_size_t()
        _check(self._lib.mla_decode_workspace_size(self._h, int(batch), int(max_ctx), ctypes.byref(out)))
        return int(out.value)

    def decode(self, q, ctx_len, max_ctx: int, block_table, cache, num_pages: int, workspace, out,
               stream=None) -> None:
        batch = int(ctx_len.shape[0])
        ws_bytes = int(workspace.numel() * workspace.element_size())
        _check(self._lib.mla_decode(self._h, _ptr(q), _ptr(ctx_len), batch, int(max_ctx), _ptr(block_table),
                                    int(block_table.shape[1]), _ptr(cache), int(num_pages), _ptr(workspace),
                                    ws_bytes, _ptr(out), _stream(stream)))

    def decode_fixed_scratch(self, q, ctx_len, max_ctx: int, block_table, cache, num_pages: int, out,
                             stream=None) -> None:
        batch = int(ctx_len.shape[0])
        _check(self._lib.mla_decode_fixed_scratch(self._h, _ptr(q), _ptr(ctx_len), batch, int(max_ctx),
                                                  _ptr(block_table), int(block_table.shape[1]), _ptr(cache),
                                                  int(num_pages), _ptr(out), _stream(stream)))

    def get_status(self, stream=None) -> int:
        flags = ctypes.c_uint32(0)
        s = self._lib.mla_get_status(self._h, _stream(stream), ctypes.byref(flags))
        if s not in (MLA_OK, MLA_ERR_DEVICE_CHECK):
            _check(s)
        return int(flags.value)

    def set_option(self, option: int, value: int) -> None:
        _check(self._lib.mla_set_option(self._h, int(option), int(value)))

    def profile_read(self) -> dict:
        buf = (ctypes.c_float * 16)()
        n = ctypes.c_int32(0)
        _check(self._lib.mla_profile_read(self._h, buf, 16, ctypes.byref(n)))
        return {self._lib.mla_profile_last_name(self._h, i).decode(): float(buf[i]) for i in range(n.value)}
