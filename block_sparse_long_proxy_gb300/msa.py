"""ctypes binding of libmsa (include/msa.h): argument marshalling only.

Every step of the hot path runs in libmsa's CUDA kernels.  Torch tensors
supply device memory and the current stream; this module checks dtypes,
shapes and contiguity, passes data_ptr()s, and raises MsaError on any
non-OK status.  Importing it fails loudly when libmsa.so is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libmsa.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_u32 = ctypes.c_uint32
_f32 = ctypes.c_float

STATUS = {0: "MSA_OK", 1: "MSA_ERR_INVALID_ARG", 2: "MSA_ERR_UNSUPPORTED", 3: "MSA_ERR_CUDA",
          4: "MSA_ERR_NO_MEMORY", 5: "MSA_ERR_TIMEOUT", 6: "MSA_ERR_DEVICE_CHECK",
          7: "MSA_ERR_NONFINITE"}
KV_BF16, KV_FP8_E4M3 = 0, 1

# Every symbol include/msa.h declares, with its ctypes signature.
SIGNATURES = {
    "msa_plan": (_i32, [_p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i64, _i32, _u32, _p, _p]),
    "msa_plan_destroy": (None, [_p]),
    "msa_plan_num_tiles": (_i32, [_p]),
    "msa_plan_max_blocks": (_i32, [_p]),
    "msa_plan_total_q": (_i64, [_p]),
    "msa_plan_num_valid_pages": (_p, [_p]),
    "msa_proxy_maxscore": (_i32, [_p, _p, _p, _p, _p, _p]),
    "msa_proxy_maxscore_fp8": (_i32, [_p, _p, _p, _p, _p, _p, _p]),
    "msa_proxy_maxscore_nvfp4": (_i32, [_p, _p, _p, _p, _p, _p, _p, _p]),
    "msa_proxy_topk": (_i32, [_p, _p, _p, _p, _p, _p, _p]),
    "msa_topk_select": (_i32, [_p, _i32, _i32, _i32, _i32, _p, _p, _p]),
    "msa_sparse_attn": (_i32, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p]),
    "msa_sparse_attn_bwd": (_i32, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _f32, _p, _p, _p, _p, _p, _p]),
    "msa_sparse_decode_noalloc": (_i32, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i64,
                                         _p, _p, _p, _p]),
    "msa_check_errors": (_i32, [_p, _p]),
    "msa_selftest_wait_timeout": (_i32, [_p]),
    "msa_test_fail_plan_allocs": (None, [_i32]),
    "msa_last_error": (ctypes.c_char_p, []),
    "msa_version": (ctypes.c_char_p, []),
}
for _name, (_res, _args) in SIGNATURES.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class MsaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _lib.msa_last_error().decode()
        super().__init__("%s: %s (%s)" % (where, STATUS.get(status, status), msg))


def _check(status, where):
    if status != 0:
        raise MsaError(status, where)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError("%s: dtype %s, want %s" % (name, t.dtype, dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s: shape %s, want %s" % (name, tuple(t.shape), tuple(shape)))
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s: must be a contiguous CUDA tensor" % name)


def version():
    return _lib.msa_version().decode()


def selftest_wait_timeout(stream=None):
    """Runs the device-side failure path once (msa_selftest_wait_timeout): a
    kernel whose bounded wait cannot complete gives up after its limit.
    Raises MsaError with status MSA_ERR_TIMEOUT, as a timed-out kernel would
    through check_errors."""
    _check(_lib.msa_selftest_wait_timeout(_stream(stream)), "msa_selftest_wait_timeout")


def inject_plan_alloc_failures(count):
    """Failure injection (msa_test_fail_plan_allocs): the next `count` plan
    creations fail at their device allocation with MSA_ERR_NO_MEMORY."""
    _lib.msa_test_fail_plan_allocs(int(count))


def topk_select(max_score, topk, num_valid_pages, out=None, stream=None):
    """kv_block_indexes [n_tiles, heads, topk] int32 from max_score [n_tiles,
    heads, max_blocks] fp32 (msa_topk_select)."""
    n, h, nb = max_score.shape
    _need(max_score, torch.float32, (n, h, nb), "max_score")
    _need(num_valid_pages, torch.int32, (n,), "num_valid_pages")
    if out is None:
        out = torch.empty((n, h, topk), dtype=torch.int32, device=max_score.device)
    _need(out, torch.int32, (n, h, topk), "kv_block_indexes")
    _check(_lib.msa_topk_select(_ptr(max_score), n, h, nb, topk, _ptr(num_valid_pages), _ptr(out),
                                _stream(stream)), "msa_topk_select")
    return out


def sparse_decode_noalloc(q, k_pages, v_pages, kv_lens, kv_indptr, kv_indices, kv_block_indexes, k_scale,
                          v_scale, out=None, lse=None, err_word=None, stream=None):
    """FP8 paged decode without a plan and without any device allocation by
    the library (msa_sparse_decode_noalloc): the batch comes as device
    int32 kv_lens [B] and kv_indptr [B+1]; scratch is libmsa's static
    array.  Outputs may be passed in (out bf16 [B, Hq, 128], lse fp32
    [B, Hq], err_word uint32/int32 [1])."""
    b, hq, d = q.shape
    hkv = k_pages.shape[1]
    topk = kv_block_indexes.shape[2]
    _need(q, torch.bfloat16, (b, hq, d), "q")
    _need(k_pages, torch.float8_e4m3fn, tuple(k_pages.shape), "k_pages")
    _need(v_pages, torch.float8_e4m3fn, tuple(k_pages.shape), "v_pages")
    _need(kv_lens, torch.int32, (b,), "kv_lens")
    _need(kv_indptr, torch.int32, (b + 1,), "kv_indptr")
    _need(kv_indices, torch.int32, (kv_indices.numel(),), "kv_indices")
    _need(kv_block_indexes, torch.int32, (b, hkv, topk), "kv_block_indexes")
    _need(k_scale, torch.float32, (hkv,), "k_scale")
    _need(v_scale, torch.float32, (hkv,), "v_scale")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, (b, hq, d), "out")
    if lse is not None:
        _need(lse, torch.float32, (b, hq), "lse")
    if err_word is not None:
        if err_word.dtype not in (torch.int32, torch.uint32) or err_word.numel() != 1:
            raise TypeError("err_word: want one 4-byte integer, got %s %s" % (err_word.dtype, tuple(err_word.shape)))
        if not err_word.is_cuda:
            raise ValueError("err_word: must be a CUDA tensor")
    _check(_lib.msa_sparse_decode_noalloc(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(kv_lens), _ptr(kv_indptr),
                                          _ptr(kv_indices), _ptr(kv_block_indexes), _ptr(k_scale), _ptr(v_scale),
                                          b, hq, hkv, d, topk, k_pages.shape[0], _ptr(out), _ptr(lse),
                                          _ptr(err_word), _stream(stream)), "msa_sparse_decode_noalloc")
    return out, lse


class Plan:
    """A validated batch shape with its device tables (msa_plan)."""

    def __init__(self, qo_lens, kv_lens, num_qo_heads, num_kv_heads, num_proxy_heads, head_dim, proxy_head_dim,
                 topk, num_pages, kv_dtype="bf16", page_size=128, stream=None):
        self.qo_lens = [int(x) for x in qo_lens]
        self.kv_lens = [int(x) for x in kv_lens]
        b = len(self.qo_lens)
        qa = (ctypes.c_int32 * b)(*self.qo_lens)
        ka = (ctypes.c_int32 * b)(*self.kv_lens)
        self.hq, self.hkv, self.hp, self.d, self.dp, self.topk = (num_qo_heads, num_kv_heads, num_proxy_heads,
                                                                  head_dim, proxy_head_dim, topk)
        self.num_pages = int(num_pages)
        self.kv_dtype = kv_dtype
        code = {"bf16": KV_BF16, "e4m3": KV_FP8_E4M3}[kv_dtype]
        h = ctypes.c_void_p()
        _check(_lib.msa_plan(qa, ka, b, num_qo_heads, num_kv_heads, num_proxy_heads, head_dim, proxy_head_dim,
                             page_size, topk, self.num_pages, code, 0, _stream(stream), ctypes.byref(h)),
               "msa_plan")
        self._h = h
        self.n_tiles = _lib.msa_plan_num_tiles(h)
        self.max_blocks = _lib.msa_plan_max_blocks(h)
        self.total_q = _lib.msa_plan_total_q(h)
        self.n_page_entries = sum((k + 127) // 128 for k in self.kv_lens)
        # a non-owning int32 view of the plan's device num_valid_pages table
        nvp_ptr = _lib.msa_plan_num_valid_pages(h)
        self._nvp_raw = nvp_ptr
        self.num_valid_pages = _device_view_int32(nvp_ptr, self.n_tiles, torch.cuda.current_device())
        self.num_valid_pages_host = None

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            _lib.msa_plan_destroy(h)
            self._h = None

    # -- stage 1
    def proxy_maxscore(self, pq, pk_pages, kv_indices, out=None, stream=None):
        _need(pq, torch.bfloat16, (self.total_q, self.hp, self.dp), "pq")
        _need(pk_pages, torch.bfloat16, (self.num_pages, 1, 128, self.dp), "pk_pages")
        _need(kv_indices, torch.int32, (self.n_page_entries,), "kv_indices")
        if out is None:
            out = torch.empty((self.n_tiles, self.hp, self.max_blocks), dtype=torch.float32, device=pq.device)
        _need(out, torch.float32, (self.n_tiles, self.hp, self.max_blocks), "max_score")
        _check(_lib.msa_proxy_maxscore(self._h, _ptr(pq), _ptr(pk_pages), _ptr(kv_indices), _ptr(out),
                                       _stream(stream)), "msa_proxy_maxscore")
        return out

    def proxy_maxscore_fp8(self, pq, pk_pages, pk_scale, kv_indices, out=None, stream=None):
        """Decode proxy pass over e4m3 proxy K pages with one fp32 scale
        (msa_proxy_maxscore_fp8)."""
        _need(pq, torch.bfloat16, (self.total_q, self.hp, self.dp), "pq")
        _need(pk_pages, torch.float8_e4m3fn, (self.num_pages, 1, 128, self.dp), "pk_pages")
        _need(pk_scale, torch.float32, (1,), "pk_scale")
        _need(kv_indices, torch.int32, (self.n_page_entries,), "kv_indices")
        if out is None:
            out = torch.empty((self.n_tiles, self.hp, self.max_blocks), dtype=torch.float32, device=pq.device)
        _need(out, torch.float32, (self.n_tiles, self.hp, self.max_blocks), "max_score")
        _check(_lib.msa_proxy_maxscore_fp8(self._h, _ptr(pq), _ptr(pk_pages), _ptr(pk_scale), _ptr(kv_indices),
                                           _ptr(out), _stream(stream)), "msa_proxy_maxscore_fp8")
        return out

    def proxy_maxscore_nvfp4(self, pq, pk_codes, pk_block_scales, pk_global_scale, kv_indices, out=None,
                             stream=None):
        """Decode proxy pass over an NVFP4 proxy K (msa_proxy_maxscore_nvfp4):
        uint8 e2m1 code pairs [P, 1, 128, dp/2], e4m3 block scales [P, 1, 128,
        dp/16] and one fp32 global scale."""
        _need(pq, torch.bfloat16, (self.total_q, self.hp, self.dp), "pq")
        _need(pk_codes, torch.uint8, (self.num_pages, 1, 128, self.dp // 2), "pk_codes")
        _need(pk_block_scales, torch.float8_e4m3fn, (self.num_pages, 1, 128, self.dp // 16), "pk_block_scales")
        _need(pk_global_scale, torch.float32, (1,), "pk_global_scale")
        _need(kv_indices, torch.int32, (self.n_page_entries,), "kv_indices")
        if out is None:
            out = torch.empty((self.n_tiles, self.hp, self.max_blocks), dtype=torch.float32, device=pq.device)
        _need(out, torch.float32, (self.n_tiles, self.hp, self.max_blocks), "max_score")
        _check(_lib.msa_proxy_maxscore_nvfp4(self._h, _ptr(pq), _ptr(pk_codes), _ptr(pk_block_scales),
                                             _ptr(pk_global_scale), _ptr(kv_indices), _ptr(out), _stream(stream)),
               "msa_proxy_maxscore_nvfp4")
        return out

    def proxy_topk(self, pq, pk_pages, kv_indices, out=None, max_score=None, stream=None):
        """Stages 1 and 2 in one launch (msa_proxy_topk): the kv_block_indexes
        msa_topk_select would pick from this plan's proxy scores; max_score,
        when given, receives those scores too."""
        _need(pq, torch.bfloat16, (self.total_q, self.hp, self.dp), "pq")
        _need(pk_pages, torch.bfloat16, (self.num_pages, 1, 128, self.dp), "pk_pages")
        _need(kv_indices, torch.int32, (self.n_page_entries,), "kv_indices")
        if out is None:
            out = torch.empty((self.n_tiles, self.hp, self.topk), dtype=torch.int32, device=pq.device)
        _need(out, torch.int32, (self.n_tiles, self.hp, self.topk), "kv_block_indexes")
        if max_score is not None:
            _need(max_score, torch.float32, (self.n_tiles, self.hp, self.max_blocks), "max_score")
        _check(_lib.msa_proxy_topk(self._h, _ptr(pq), _ptr(pk_pages), _ptr(kv_indices), _ptr(max_score), _ptr(out),
                                   _stream(stream)), "msa_proxy_topk")
        return out

    # -- stage 3
    def sparse_attn(self, q, k_pages, v_pages, kv_indices, kv_block_indexes, k_scale=None, v_scale=None,
                    out=None, lse=None, want_lse=True, stream=None):
        _need(q, torch.bfloat16, (self.total_q, self.hq, self.d), "q")
        kvt = torch.bfloat16 if self.kv_dtype == "bf16" else torch.float8_e4m3fn
        _need(k_pages, kvt, (self.num_pages, self.hkv, 128, self.d), "k_pages")
        _need(v_pages, kvt, (self.num_pages, self.hkv, 128, self.d), "v_pages")
        _need(kv_indices, torch.int32, (self.n_page_entries,), "kv_indices")
        _need(kv_block_indexes, torch.int32, (self.n_tiles, self.hp, self.topk), "kv_block_indexes")
        if self.kv_dtype != "bf16":
            _need(k_scale, torch.float32, (self.hkv,), "k_scale")
            _need(v_scale, torch.float32, (self.hkv,), "v_scale")
        if out is None:
            out = torch.empty_like(q)
        _need(out, torch.bfloat16, tuple(q.shape), "out")
        if lse is None and want_lse:
            lse = torch.empty((self.total_q, self.hq), dtype=torch.float32, device=q.device)
        if lse is not None:
            _need(lse, torch.float32, (self.total_q, self.hq), "lse")
        _check(_lib.msa_sparse_attn(self._h, _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(kv_indices),
                                    _ptr(kv_block_indexes), _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(lse),
                                    _stream(stream)), "msa_sparse_attn")
        return out, lse

    # -- training extension
    def sparse_attn_bwd(self, q, k_pages, v_pages, kv_indices, kv_block_indexes, out, lse, dout, pq, pk_pages,
                        kl_weight=1.0, grads=None, stream=None):
        _need(dout, torch.bfloat16, tuple(q.shape), "dout")
        _need(out, torch.bfloat16, tuple(q.shape), "out")
        _need(lse, torch.float32, (self.total_q, self.hq), "lse")
        _need(pq, torch.bfloat16, (self.total_q, self.hp, self.dp), "pq")
        _need(pk_pages, torch.bfloat16, (self.num_pages, 1, 128, self.dp), "pk_pages")
        _need(kv_block_indexes, torch.int32, (self.n_tiles, self.hp, self.topk), "kv_block_indexes")
        dev = q.device
        if grads is None:
            grads = dict(dq=torch.empty(q.shape, dtype=torch.float32, device=dev),
                         dk=torch.zeros(k_pages.shape, dtype=torch.float32, device=dev),
                         dv=torch.zeros(v_pages.shape, dtype=torch.float32, device=dev),
                         dpq=torch.empty(pq.shape, dtype=torch.float32, device=dev),
                         dpk=torch.zeros(pk_pages.shape, dtype=torch.float32, device=dev))
        _check(_lib.msa_sparse_attn_bwd(self._h, _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(kv_indices),
                                        _ptr(kv_block_indexes), _ptr(out), _ptr(lse), _ptr(dout), _ptr(pq),
                                        _ptr(pk_pages), float(kl_weight), _ptr(grads["dq"]), _ptr(grads["dk"]),
                                        _ptr(grads["dv"]), _ptr(grads["dpq"]), _ptr(grads["dpk"]),
                                        _stream(stream)), "msa_sparse_attn_bwd")
        return grads

    def check_errors(self, stream=None):
        _check(_lib.msa_check_errors(self._h, _stream(stream)), "msa_check_errors")


def _device_view_int32(ptr, n, device_index):
    """Wrap a device int32 array owned by libmsa as a torch tensor without
    copying (the plan keeps it alive)."""
    class _Holder:
        pass
    h = _Holder()
    h.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (ptr, False), "version": 3,
                                  "strides": None}
    with torch.cuda.device(device_index):
        return torch.as_tensor(h, device="cuda:%d" % device_index)
