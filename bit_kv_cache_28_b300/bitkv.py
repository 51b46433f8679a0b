"""ctypes binding of libbitkv.so (declared in include/bitkv.h).

Argument marshalling only: every call goes straight to the C ABI, and every
step of the path runs in the library's CUDA kernels.  PyTorch is used for
device memory and streams (``TorchCache`` allocates a cache's regions with
``torch.empty``).  Loading fails loudly if the library has not been built;
there is no fallback.
"""

from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libbitkv.so")

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_UNSUPPORTED, KV_ERR_CAPACITY = 0, 1, 2, 3
KV_ERR_WORKSPACE, KV_ERR_ALIGNMENT, KV_ERR_CUDA, KV_ERR_TIMEOUT, KV_ERR_RANGE = 4, 5, 6, 7, 8
KV_F32, KV_F16, KV_BF16 = 0, 1, 2
KV_UNIFORM2, KV_UNIFORM4, KV_MIXED, KV_CODEBOOK2 = 0, 1, 2, 3
KV_SEG_RAW16, KV_SEG_INT4, KV_SEG_INT2 = 0, 1, 2
KV_REGION_DATA, KV_REGION_BLK_LEN, KV_REGION_BLK_POS, KV_REGION_CENTROIDS, KV_REGION_PSAC_U = 0, 1, 2, 3, 4
KV_REGION_RESID_VAR = 5
KV_JENSEN_OFF, KV_JENSEN_TAYLOR2, KV_JENSEN_EXACT, KV_JENSEN_ISOTROPIC = 0, 1, 2, 3
KV_PATH_AUTO, KV_PATH_SIMT, KV_PATH_TC, KV_PATH_DECODE, KV_PATH_TC_SINGLE = 0, 1, 2, 3, 4

STATUS_NAMES = {0: "KV_OK", 1: "KV_ERR_INVALID_ARG", 2: "KV_ERR_UNSUPPORTED", 3: "KV_ERR_CAPACITY",
                4: "KV_ERR_WORKSPACE", 5: "KV_ERR_ALIGNMENT", 6: "KV_ERR_CUDA", 7: "KV_ERR_TIMEOUT",
                8: "KV_ERR_RANGE"}

# Every symbol the header declares (checked by the CPU test suite).
EXPORTS = ["kv_layout_init", "kv_layout_bytes", "kv_cache_init", "kv_quantize_append", "kv_attention_workspace",
           "kv_attention_plan", "kv_attention", "kv_attention_status", "kv_attention_noalloc",
           "kv_attention_noalloc_status", "kv_window_plan", "kv_window_similarity",
           "kv_codebook_workspace", "kv_codebook_fit", "kv_codebook_fit_range", "kv_codebook_residual_var",
           "kv_psac_workspace",
           "kv_psac_basis", "kv_dequantize", "kv_debug_operands", "kv_last_error", "kv_version"]


class kv_layout(C.Structure):
    _fields_ = [("B", C.c_int32), ("Hkv", C.c_int32), ("d", C.c_int32), ("kind", C.c_int32),
                ("raw_dtype", C.c_int32), ("psac_rank", C.c_int32), ("cap_blocks", C.c_int32 * 3),
                ("meta_dtype", C.c_int32), ("block_bytes", C.c_int64 * 3), ("seg_offset", C.c_int64 * 3), ("stream_bytes", C.c_int64)]


class kv_cache(C.Structure):
    _fields_ = [("layout", kv_layout), ("data", C.c_void_p), ("blk_len", C.c_void_p), ("blk_pos", C.c_void_p),
                ("centroids", C.c_void_p), ("psac_u", C.c_void_p), ("n_blocks", C.c_int32 * 3),
                ("n_tokens", C.c_int32), ("resid_var", C.c_void_p)]


class kv_append_opts(C.Structure):
    _fields_ = [("window_bits_host", C.c_void_p), ("window_bits_dev", C.c_void_p)]


class kv_attn_opts(C.Structure):
    _fields_ = [("scale", C.c_float), ("jensen", C.c_int32), ("psac", C.c_int32), ("out_f32", C.c_int32),
                ("num_splits", C.c_int32), ("path", C.c_int32)]


class kv_thresholds(C.Structure):
    _fields_ = [("frac_fp16", C.c_double), ("frac_int4", C.c_double), ("force_first", C.c_int32)]


class BitKVError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib():
    """Load libbitkv.so (raises if it is missing: there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"libbitkv.so not built ({_LIB_PATH}); run __graft_entry__.build()")
        L = C.CDLL(_LIB_PATH)
        P, I, S = C.c_void_p, C.c_int, C.c_size_t
        sig = {
            "kv_layout_init": (C.c_int, [C.POINTER(kv_layout), I, I, I, I, I, C.POINTER(C.c_int32), I, I]),
            "kv_layout_bytes": (S, [C.POINTER(kv_layout), I]),
            "kv_cache_init": (C.c_int, [C.POINTER(kv_cache), C.POINTER(kv_layout), P, P, P, P, P]),
            "kv_quantize_append": (C.c_int, [P, P, I, I, C.POINTER(kv_cache), C.POINTER(kv_append_opts), P]),
            "kv_attention_workspace": (S, [C.POINTER(kv_cache), I, I, I, I, C.POINTER(kv_attn_opts)]),
            "kv_attention_plan": (C.c_int, [C.POINTER(kv_cache), I, I, I, I, C.POINTER(kv_attn_opts),
                                            C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
            "kv_attention": (C.c_int, [P, P, P, I, I, I, I, C.POINTER(kv_cache), C.POINTER(kv_attn_opts), P, P, P, S, P]),
            "kv_attention_status": (C.c_int, [P, P]),
            "kv_attention_noalloc": (C.c_int, [P, P, P, I, I, I, I, C.POINTER(kv_cache), C.POINTER(kv_attn_opts), P,
                                               P, P]),
            "kv_attention_noalloc_status": (C.c_int, [P]),
            "kv_window_plan": (C.c_int, [P, I, C.POINTER(kv_thresholds), P, P]),
            "kv_window_similarity": (C.c_int, [P, P, I, I, I, I, I, I, P, P]),
            "kv_codebook_workspace": (S, [C.POINTER(kv_layout), I]),
            "kv_codebook_fit": (C.c_int, [P, I, I, C.POINTER(kv_cache), I, P, I, P, P, S, P]),
            "kv_codebook_fit_range": (C.c_int, [P, I, I, C.POINTER(kv_cache), I, P, I, P, P]),
            "kv_codebook_residual_var": (C.c_int, [P, I, I, C.POINTER(kv_cache), P]),
            "kv_psac_workspace": (S, [C.POINTER(kv_layout)]),
            "kv_psac_basis": (C.c_int, [P, I, I, C.POINTER(kv_cache), P, P, S, P]),
            "kv_dequantize": (C.c_int, [C.POINTER(kv_cache), P, P, P]),
            "kv_debug_operands": (C.c_int, [C.POINTER(kv_cache), I, P, P, P]),
            "kv_last_error": (C.c_char_p, []),
            "kv_version": (C.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status):
    if status != KV_OK:
        raise BitKVError(status, lib().kv_last_error().decode())


def _ptr(x):
    """Device/host address of a torch tensor, numpy array, int or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(type(x))


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- calls ----

def kv_layout_init(B, Hkv, d, kind, raw_dtype=KV_F16, cap_blocks=(0, 0, 0), psac_rank=0,
                   meta_dtype=KV_F32) -> kv_layout:
    L = kv_layout()
    caps = (C.c_int32 * 3)(*cap_blocks)
    _check(lib().kv_layout_init(C.byref(L), B, Hkv, d, kind, raw_dtype, caps, psac_rank, meta_dtype))
    return L


def kv_layout_bytes(layout: kv_layout, region: int) -> int:
    return int(lib().kv_layout_bytes(C.byref(layout), region))


def kv_cache_init(layout, data, blk_len, blk_pos, centroids=None, psac_u=None) -> kv_cache:
    c = kv_cache()
    _check(lib().kv_cache_init(C.byref(c), C.byref(layout), _ptr(data), _ptr(blk_len), _ptr(blk_pos),
                               _ptr(centroids), _ptr(psac_u)))
    return c


def kv_quantize_append(K, V, dtype, n_tokens, cache: kv_cache, opts: kv_append_opts | None = None, stream=None):
    _check(lib().kv_quantize_append(_ptr(K), _ptr(V), dtype, n_tokens, C.byref(cache),
                                    C.byref(opts) if opts is not None else None, _stream(stream)))


def kv_attention_workspace(cache, dtype, n_q, n_cur, Hq, opts: kv_attn_opts | None = None) -> int:
    return int(lib().kv_attention_workspace(C.byref(cache), dtype, n_q, n_cur, Hq,
                                            C.byref(opts) if opts is not None else None))


def kv_attention_plan(cache, dtype, n_q, n_cur, Hq, opts: kv_attn_opts | None = None):
    """(path, splits) kv_attention would use; launches nothing."""
    path, splits = C.c_int32(0), C.c_int32(0)
    _check(lib().kv_attention_plan(C.byref(cache), dtype, n_q, n_cur, Hq,
                                   C.byref(opts) if opts is not None else None, C.byref(path), C.byref(splits)))
    return path.value, splits.value


def kv_attention(Q, Kcur, Vcur, dtype, n_q, n_cur, Hq, cache, opts, out, lse=None, workspace=None, ws_bytes=0,
                 stream=None):
    _check(lib().kv_attention(_ptr(Q), _ptr(Kcur), _ptr(Vcur), dtype, n_q, n_cur, Hq, C.byref(cache),
                              C.byref(opts) if opts is not None else None, _ptr(out), _ptr(lse), _ptr(workspace),
                              ws_bytes, _stream(stream)))


def kv_attention_status(workspace, stream=None):
    """Raises BitKVError if the last kv_attention on `workspace` timed out or hit the fp16 range."""
    _check(lib().kv_attention_status(_ptr(workspace), _stream(stream)))


def kv_attention_noalloc_status(stream=None):
    """kv_attention_status for the last kv_attention_noalloc call on the current device."""
    _check(lib().kv_attention_noalloc_status(_stream(stream)))


def kv_attention_noalloc(Q, Kcur, Vcur, dtype, n_q, n_cur, Hq, cache, opts, out, lse=None, stream=None):
    """kv_attention with its scratch in the library's fixed device array (no workspace argument)."""
    _check(lib().kv_attention_noalloc(_ptr(Q), _ptr(Kcur), _ptr(Vcur), dtype, n_q, n_cur, Hq, C.byref(cache),
                                      C.byref(opts) if opts is not None else None, _ptr(out), _ptr(lse),
                                      _stream(stream)))


def kv_window_plan(sim, n_windows, thresholds: kv_thresholds | None, bits_out, perm_out=None):
    """Host-only: sim, bits_out (int8) and perm_out (int32) are numpy arrays."""
    _check(lib().kv_window_plan(_ptr(sim), n_windows, C.byref(thresholds) if thresholds is not None else None,
                                _ptr(bits_out), _ptr(perm_out)))


def kv_window_similarity(K, Kq, dtype, B, Hkv, n, m, d, sim, stream=None):
    """Device: K [B][Hkv][n][d], Kq [B][Hkv][m][d] in dtype; sim fp32 [B][ceil(n / 32)]."""
    _check(lib().kv_window_similarity(_ptr(K), _ptr(Kq), dtype, B, Hkv, n, m, d, _ptr(sim), _stream(stream)))


def kv_codebook_workspace(layout, n_tokens) -> int:
    return int(lib().kv_codebook_workspace(C.byref(layout), n_tokens))


def kv_codebook_fit(K, dtype, n_tokens, cache, iters=20, Qhist=None, n_hist=0, weights_out=None, workspace=None,
                    ws_bytes=0, stream=None):
    _check(lib().kv_codebook_fit(_ptr(K), dtype, n_tokens, C.byref(cache), iters, _ptr(Qhist), n_hist,
                                 _ptr(weights_out), _ptr(workspace), ws_bytes, _stream(stream)))


def kv_codebook_fit_range(K, dtype, n_tokens, cache, iters, Qhist, n_hist, weights_out, stream=None):
    _check(lib().kv_codebook_fit_range(_ptr(K), dtype, n_tokens, C.byref(cache), iters, _ptr(Qhist), n_hist,
                                       _ptr(weights_out), _stream(stream)))


def kv_codebook_residual_var(K, dtype, n_tokens, cache, stream=None):
    _check(lib().kv_codebook_residual_var(_ptr(K), dtype, n_tokens, C.byref(cache), _stream(stream)))


def kv_psac_workspace(layout) -> int:
    return int(lib().kv_psac_workspace(C.byref(layout)))


def kv_psac_basis(Qhist, dtype, n_hist, cache, eigvals_out=None, workspace=None, ws_bytes=0, stream=None):
    _check(lib().kv_psac_basis(_ptr(Qhist), dtype, n_hist, C.byref(cache), _ptr(eigvals_out), _ptr(workspace),
                               ws_bytes, _stream(stream)))


def kv_dequantize(cache, K_out, V_out, stream=None):
    _check(lib().kv_dequantize(C.byref(cache), _ptr(K_out), _ptr(V_out), _stream(stream)))


def kv_debug_operands(cache, path, K_out, V_out, stream=None):
    """The fp16 cache operands the tensor-core (KV_PATH_TC) or decode (KV_PATH_DECODE) kernel builds."""
    _check(lib().kv_debug_operands(C.byref(cache), path, _ptr(K_out), _ptr(V_out), _stream(stream)))


def kv_last_error() -> str:
    return lib().kv_last_error().decode()


def kv_version() -> str:
    return lib().kv_version().decode()


# ------------------------------------------------------- torch plumbing ----

def torch_dtype_code(t):
    import torch
    return {torch.float32: KV_F32, torch.float16: KV_F16, torch.bfloat16: KV_BF16}[t]


class TorchCache:
    """A cache whose regions are torch tensors on one CUDA device (allocation only)."""

    def __init__(self, B, Hkv, d, kind, cap_blocks, raw_dtype=KV_F16, psac_rank=0, device="cuda", resid_var=False,
                 meta_dtype=KV_F32):
        import torch
        self.layout = kv_layout_init(B, Hkv, d, kind, raw_dtype, cap_blocks, psac_rank, meta_dtype)
        nb = lambda r: kv_layout_bytes(self.layout, r)
        self.data = torch.zeros(nb(KV_REGION_DATA), dtype=torch.uint8, device=device)
        self.blk_len = torch.zeros(max(1, nb(KV_REGION_BLK_LEN) // 4), dtype=torch.int32, device=device)
        self.blk_pos = torch.zeros(max(1, nb(KV_REGION_BLK_POS) // 4), dtype=torch.int32, device=device)
        self.centroids = (torch.zeros(nb(KV_REGION_CENTROIDS) // 4, dtype=torch.float32, device=device)
                          if nb(KV_REGION_CENTROIDS) else None)
        self.psac_u = (torch.zeros(nb(KV_REGION_PSAC_U) // 4, dtype=torch.float32, device=device)
                       if nb(KV_REGION_PSAC_U) else None)
        self.c = kv_cache_init(self.layout, self.data, self.blk_len, self.blk_pos, self.centroids, self.psac_u)
        # CODEBOOK2: the keys' residual variances, which turn on their Jensen term
        self.resid_var = None
        if resid_var and nb(KV_REGION_RESID_VAR):
            self.resid_var = torch.zeros(nb(KV_REGION_RESID_VAR) // 4, dtype=torch.float32, device=device)
            self.c.resid_var = self.resid_var.data_ptr()

    @property
    def n_tokens(self):
        return self.c.n_tokens

    @property
    def n_blocks(self):
        return list(self.c.n_blocks)

    def reset(self):
        """Forget all appended tokens (host counters only; bytes stay until overwritten)."""
        self.c.n_tokens = 0
        for i in range(3):
            self.c.n_blocks[i] = 0
