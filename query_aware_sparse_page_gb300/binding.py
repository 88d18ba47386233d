"""ctypes binding of libspg.so: argument marshalling only.

Every function here has the name of the C entry point it calls, checks that
the tensors it is given are contiguous CUDA tensors, passes their device
pointers and the current CUDA stream, and turns a non-OK status into
SpgError.  No step of the computation runs in Python, and there is no
fallback: if the library is missing, importing this module fails.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_size_t, c_void_p

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspg.so")

SPG_OK, SPG_EINVAL, SPG_EUNSUPPORTED, SPG_ECUDA, SPG_EWORKSPACE = 0, 1, 2, 3, 4
SEL_QUEST, SEL_SKETCH_INT4, SEL_ALL, SEL_PROBE = 0, 1, 2, 3
F16, BF16, I8 = 0, 1, 2
DEVERR_PAGE_ID, DEVERR_SEQ_LEN, DEVERR_SEL, DEVERR_TIMEOUT = 1, 2, 4, 8

_DTYPES = {"f16": F16, "bf16": BF16, "i8": I8}
_SELECTORS = {"quest": SEL_QUEST, "sketch": SEL_SKETCH_INT4, "all": SEL_ALL, "probe": SEL_PROBE}


class SpgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} (status {status})")


class spg_params(ctypes.Structure):
    _fields_ = [
        ("batch", c_int32),
        ("num_q_heads", c_int32),
        ("num_kv_heads", c_int32),
        ("head_dim", c_int32),
        ("page_size", c_int32),
        ("num_phys_pages", c_int32),
        ("max_pages_per_seq", c_int32),
        ("kv_dtype", c_int32),
        ("q_dtype", c_int32),
        ("selector", c_int32),
        ("token_budget", c_int32),
        ("n_sink_pages", c_int32),
        ("n_recent_pages", c_int32),
        ("sketch_dim", c_int32),
        ("softmax_scale", c_float),
        ("top_p", c_float),
        ("min_pages", c_int32),
        ("n_probe", c_int32),
    ]

    def __repr__(self):
        return "spg_params(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


def make_params(batch, num_q_heads, num_kv_heads, head_dim, page_size, num_phys_pages,
                max_pages_per_seq, kv_dtype="f16", q_dtype=None, selector="quest",
                token_budget=0, n_sink_pages=0, n_recent_pages=0, sketch_dim=16,
                softmax_scale=0.0, top_p=0.0, min_pages=0, n_probe=0) -> spg_params:
    kv = _DTYPES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
    if q_dtype is None:
        q_dtype = kv if kv != I8 else F16
    qd = _DTYPES[q_dtype] if isinstance(q_dtype, str) else int(q_dtype)
    sel = _SELECTORS[selector] if isinstance(selector, str) else int(selector)
    return spg_params(batch, num_q_heads, num_kv_heads, head_dim, page_size, num_phys_pages,
                      max_pages_per_seq, kv, qd, sel, token_budget, n_sink_pages, n_recent_pages,
                      sketch_dim, softmax_scale, top_p, min_pages, n_probe)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run query_aware_sparse_page_gb300._build.build() "
            "(nvcc for sm_103a).  There is no fallback implementation.")
    lib = ctypes.CDLL(LIB_PATH)
    P = POINTER(spg_params)
    v = c_void_p
    sigs = {
        "spg_abi_version": ([], c_int32),
        "spg_status_str": ([c_int32], c_char_p),
        "spg_validate": ([P], c_int32),
        "spg_workspace_size": ([P, POINTER(c_size_t)], c_int32),
        "sparse_page_meta_update": ([P, v, v, v, v, c_int32, v, v, v, v, v, c_size_t, v], c_int32),
        "sparse_page_score": ([P, v, v, v, v, v, v, v, v, v, c_size_t, v], c_int32),
        "sparse_page_select": ([P, v, v, v, v, v, v, v, v, v, v, c_size_t, v], c_int32),
        "sparse_decode_attention": ([P, v, v, v, v, v, v, v, v, v, v, v, v, c_size_t, v], c_int32),
        "sparse_decode_select_attend": (
            [P, v, v, v, v, v, v, v, v, v, v, v, v, v, v, v, v, c_size_t, v], c_int32),
        "dense_decode_attention": ([P, v, v, v, v, v, v, v, v, v, v, c_size_t, v], c_int32),
        "sparse_decode_step": (
            [P, v, v, v, v, v, v, v, v, v, v, v, v, v, v, v, v, c_size_t, v], c_int32),
        "sparse_page_sketch_dots": ([P, v, v, v, v, v, v, v, v, c_size_t, v], c_int32),
        "spg_step_kernel": ([P], c_char_p),
        "spg_prefer_dense": ([P, c_int32, c_float], c_int32),
        "spg_step_launches": ([P], c_int32),
        "spg_set_step_kernel": ([c_int32], c_int32),
        "spg_read_device_error": ([v, POINTER(c_int32), v], c_int32),
        "spg_clear_device_error": ([v, v], c_int32),
        "spg_test_withhold_first_stage": ([v, v], c_int32),
    }
    for name, (args, res) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


LIB = _load()


# ---- marshalling helpers ----------------------------------------------------
def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libspg takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libspg takes contiguous tensors")
    return c_void_p(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return c_void_p(int(stream))
    import torch

    return c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status: int, where: str):
    if status != SPG_OK:
        raise SpgError(status, where)


def _ws(ws):
    return _ptr(ws), c_size_t(ws.numel() * ws.element_size())


# ---- host-only entry points ---------------------------------------------------
def spg_abi_version() -> int:
    return LIB.spg_abi_version()


def status_str(status: int) -> str:
    return LIB.spg_status_str(status).decode()


spg_status_str = status_str


def spg_validate(p: spg_params) -> int:
    return LIB.spg_validate(ctypes.byref(p))


def spg_workspace_size(p: spg_params) -> int:
    n = c_size_t(0)
    _check(LIB.spg_workspace_size(ctypes.byref(p), ctypes.byref(n)), "spg_workspace_size")
    return n.value


def spg_step_kernel(p: spg_params) -> str | None:
    r = LIB.spg_step_kernel(ctypes.byref(p))
    return None if r is None else r.decode()


step_kernel_name = spg_step_kernel


def spg_prefer_dense(p: spg_params, max_seq_len: int, ratio: float = 0.0) -> bool:
    return bool(LIB.spg_prefer_dense(ctypes.byref(p), int(max_seq_len), float(ratio)))


def spg_step_launches(p: spg_params) -> int:
    return LIB.spg_step_launches(ctypes.byref(p))


step_launch_count = spg_step_launches

STEP_KERNEL_AUTO, STEP_KERNEL_CLUSTER, STEP_KERNEL_SCHED = 0, 1, 2


def spg_set_step_kernel(kernel: int):
    _check(LIB.spg_set_step_kernel(int(kernel)), "spg_set_step_kernel")


# ---- device entry points -------------------------------------------------------
def sparse_page_meta_update(p, k_pool, k_scale, page_table, seq_lens, rebuild, minmax=None,
                            sketch=None, sketch_scale=None, proj=None, ws=None, stream=None):
    wp, wn = _ws(ws)
    _check(LIB.sparse_page_meta_update(
        ctypes.byref(p), _ptr(k_pool), _ptr(k_scale), _ptr(page_table), _ptr(seq_lens),
        int(rebuild), _ptr(minmax), _ptr(sketch), _ptr(sketch_scale), _ptr(proj), wp, wn,
        _stream(stream)), "sparse_page_meta_update")


def sparse_page_score(p, q, page_table, seq_lens, minmax=None, sketch=None, sketch_scale=None,
                      proj=None, scores=None, ws=None, stream=None):
    wp, wn = _ws(ws)
    _check(LIB.sparse_page_score(
        ctypes.byref(p), _ptr(q), _ptr(page_table), _ptr(seq_lens), _ptr(minmax), _ptr(sketch),
        _ptr(sketch_scale), _ptr(proj), _ptr(scores), wp, wn, _stream(stream)),
        "sparse_page_score")


def sparse_page_sketch_dots(p, q, seq_lens, sketch, proj, qc, sq, dots, ws, stream=None):
    wp, wn = _ws(ws)
    _check(LIB.sparse_page_sketch_dots(
        ctypes.byref(p), _ptr(q), _ptr(seq_lens), _ptr(sketch), _ptr(proj), _ptr(qc), _ptr(sq),
        _ptr(dots), wp, wn, _stream(stream)), "sparse_page_sketch_dots")


def sparse_page_select(p, q, page_table, seq_lens, minmax=None, sketch=None, sketch_scale=None,
                       proj=None, sel=None, sel_cnt=None, ws=None, stream=None):
    wp, wn = _ws(ws)
    _check(LIB.sparse_page_select(
        ctypes.byref(p), _ptr(q), _ptr(page_table), _ptr(seq_lens), _ptr(minmax), _ptr(sketch),
        _ptr(sketch_scale), _ptr(proj), _ptr(sel), _ptr(sel_cnt), wp, wn, _stream(stream)),
        "sparse_page_select")


def sparse_decode_attention(p, q, k_pool, v_pool, k_scale, v_scale, page_table, seq_lens, sel,
                            sel_cnt, out, lse=None, ws=None, stream=None):
    wp, wn = _ws(ws)
    _check(LIB.sparse_decode_attention(
        ctypes.byref(p), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
        _ptr(page_table), _ptr(seq_lens), _ptr(sel), _ptr(sel_cnt), _ptr(out), _ptr(lse), wp, wn,
        _stream(stream)), "sparse_decode_attention")


def sparse_decode_select_attend(p, q, k_pool, v_pool, k_scale, v_scale, page_table, seq_lens,
                                minmax=None, sketch=None, sketch_scale=None, proj=None, sel=None,
                                sel_cnt=None, out=None, lse=None, ws=None, stream=None):
    wp, wn = _ws(ws)
    _check(LIB.sparse_decode_select_attend(
        ctypes.byref(p), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
        _ptr(page_table), _ptr(seq_lens), _ptr(minmax), _ptr(sketch), _ptr(sketch_scale),
        _ptr(proj), _ptr(sel), _ptr(sel_cnt), _ptr(out), _ptr(lse), wp, wn, _stream(stream)),
        "sparse_decode_select_attend")


def sparse_decode_step(p, q, k_pool, v_pool, k_scale, v_scale, page_table, seq_lens,
                       minmax=None, sketch=None, sketch_scale=None, proj=None, sel=None,
                       sel_cnt=None, out=None, lse=None, ws=None, stream=None):
    wp, wn = _ws(ws)
    _check(LIB.sparse_decode_step(
        ctypes.byref(p), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
        _ptr(page_table), _ptr(seq_lens), _ptr(minmax), _ptr(sketch), _ptr(sketch_scale),
        _ptr(proj), _ptr(sel), _ptr(sel_cnt), _ptr(out), _ptr(lse), wp, wn, _stream(stream)),
        "sparse_decode_step")


def dense_decode_attention(p, q, k_pool, v_pool, k_scale, v_scale, page_table, seq_lens, out,
                           lse=None, ws=None, stream=None):
    wp, wn = _ws(ws)
    _check(LIB.dense_decode_attention(
        ctypes.byref(p), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
        _ptr(page_table), _ptr(seq_lens), _ptr(out), _ptr(lse), wp, wn, _stream(stream)),
        "dense_decode_attention")


def spg_read_device_error(ws, stream=None) -> int:
    bits = c_int32(0)
    _check(LIB.spg_read_device_error(_ptr(ws), ctypes.byref(bits), _stream(stream)),
           "spg_read_device_error")
    return bits.value


def spg_clear_device_error(ws, stream=None):
    _check(LIB.spg_clear_device_error(_ptr(ws), _stream(stream)), "spg_clear_device_error")


def spg_test_withhold_first_stage(ws, stream=None):
    _check(LIB.spg_test_withhold_first_stage(_ptr(ws), _stream(stream)), "spg_test_withhold_first_stage")
