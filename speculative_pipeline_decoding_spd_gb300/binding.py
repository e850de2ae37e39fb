"""ctypes binding of include/spd.h: the same names and arguments, marshalling only.

All computation happens in libspd_gb300.so; this module converts Python values into the
ABI's structs and pointers.  Loading fails loudly when the library has not been built:
there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspd_gb300.so")

SPD_OK, SPD_EINVAL, SPD_ENOMEM, SPD_ECUDA, SPD_ESTATE, SPD_ECAPACITY, SPD_EDEVICE = range(7)
SPD_F32, SPD_BF16, SPD_F16 = 0, 1, 2
SPD_SPEC_INPUT, SPD_SPEC_OUTPUT = 0, 1
SPD_MAX_ANCHORS, SPD_MAX_STAGES, SPD_MAX_LAYERS, SPD_MAX_PDM_LAYERS = 8, 31, 128, 16
(SPD_BUF_RESIDUAL, SPD_BUF_ANCHORS, SPD_BUF_LOGITS, SPD_BUF_KCACHE, SPD_BUF_VCACHE, SPD_BUF_PDM_KCACHE,
 SPD_BUF_PDM_VCACHE, SPD_BUF_SLOTS, SPD_BUF_STATE, SPD_BUF_PREFILL_LOGITS, SPD_BUF_PDM_RESIDUAL) = range(11)

ERRORS = {SPD_EINVAL: "EINVAL", SPD_ENOMEM: "ENOMEM", SPD_ECUDA: "ECUDA", SPD_ESTATE: "ESTATE",
          SPD_ECAPACITY: "ECAPACITY", SPD_EDEVICE: "EDEVICE"}


class spd_dims(C.Structure):
    _fields_ = [("L", C.c_int32), ("d", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32), ("hd", C.c_int32),
                ("F", C.c_int32), ("V", C.c_int32), ("rope_theta", C.c_float), ("rms_eps", C.c_float),
                ("dtype", C.c_int32)]


class spd_layer_weights(C.Structure):
    _fields_ = [("wq", C.c_void_p), ("wk", C.c_void_p), ("wv", C.c_void_p), ("wo", C.c_void_p),
                ("w_gate", C.c_void_p), ("w_up", C.c_void_p), ("w_down", C.c_void_p),
                ("attn_norm", C.c_void_p), ("ffn_norm", C.c_void_p)]


class spd_target_weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("layers", C.POINTER(spd_layer_weights)), ("final_norm", C.c_void_p),
                ("lm_head", C.c_void_p)]


class spd_pdm_weights(C.Structure):
    _fields_ = [("Ls", C.c_int32), ("proj", C.c_void_p), ("layers", C.POINTER(spd_layer_weights)),
                ("final_norm", C.c_void_p), ("lm_head", C.c_void_p)]


class spd_config(C.Structure):
    _fields_ = [("n", C.c_int32), ("n_anchors", C.c_int32), ("anchors", C.c_int32 * SPD_MAX_ANCHORS),
                ("temperature", C.c_float), ("seed", C.c_uint64), ("max_seq", C.c_int32), ("max_new", C.c_int32),
                ("force_p", C.c_float), ("forced_ref", C.c_void_p), ("forced_ref_len", C.c_int32),
                ("graph", C.c_int32), ("timing", C.c_int32), ("stage_bounds", C.c_int32 * (SPD_MAX_STAGES + 1)),
                ("speculate", C.c_int32)]


class spd_stats(C.Structure):
    _fields_ = [("N", C.c_int64), ("K", C.c_int64), ("accepts", C.c_int64), ("rejects", C.c_int64),
                ("alpha", C.c_double), ("S0", C.c_double), ("mean_kept_run", C.c_double),
                ("weight_bytes", C.c_double), ("ls_exceeds_masking", C.c_int32), ("device_error", C.c_int32)]


class spd_trace_rec(C.Structure):
    _fields_ = [("t", C.c_int32), ("exit_pos", C.c_int32), ("draft", C.c_int32), ("target", C.c_int32),
                ("accept", C.c_int32), ("commit", C.c_int32), ("pdm_top", C.c_int32), ("new_draft", C.c_int32),
                ("n_committed", C.c_int32), ("n_active", C.c_int32), ("target_logit", C.c_float),
                ("pdm_logit", C.c_float)]


class spd_trace_view(C.Structure):
    _fields_ = [("recs", C.c_void_p), ("kv_len", C.c_void_p), ("count", C.c_int32), ("L", C.c_int32)]


_lib = None

# (name, restype, argtypes) of every entry point declared in include/spd.h
SIGNATURES = [
    ("spd_workspace_bytes", C.c_int, [C.POINTER(spd_dims), C.POINTER(spd_pdm_weights), C.POINTER(spd_config),
                                      C.POINTER(C.c_size_t)]),
    ("spd_create", C.c_int, [C.POINTER(spd_dims), C.POINTER(spd_target_weights), C.POINTER(spd_pdm_weights),
                             C.POINTER(spd_config), C.c_void_p, C.c_size_t, C.c_void_p, C.POINTER(C.c_void_p)]),
    ("spd_prefill", C.c_int, [C.c_void_p, C.c_void_p, C.c_int32]),
    ("spd_step", C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int32)]),
    ("spd_generate", C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.POINTER(C.c_int32),
                               C.POINTER(spd_stats)]),
    ("spd_get_trace", C.c_int, [C.c_void_p, C.POINTER(spd_trace_rec), C.c_int32, C.c_void_p, C.POINTER(C.c_int32)]),
    ("spd_get_trace_view", C.c_int, [C.c_void_p, C.POINTER(spd_trace_view)]),
    ("spd_get_stats", C.c_int, [C.c_void_p, C.POINTER(spd_stats)]),
    ("spd_get_tokens", C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.POINTER(C.c_int32)]),
    ("spd_read_buffer", C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_size_t, C.c_void_p, C.c_size_t]),
    ("spd_kernel_timing", C.c_int, [C.c_void_p, C.POINTER(C.c_double), C.POINTER(C.c_int64)]),
    ("spd_attention_scratch_bytes", C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.POINTER(C.c_size_t)]),
    ("spd_attention_decode", C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                       C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    ("spd_attention_decode_noalloc", C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                               C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    ("spd_ops_last_error", C.c_char_p, []),
    ("spd_reset", C.c_int, [C.c_void_p]),
    ("spd_destroy", None, [C.c_void_p]),
    ("spd_last_error", C.c_char_p, [C.c_void_p]),
]


def load(path: str = LIB_PATH):
    """Load libspd_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m speculative_pipeline_decoding_spd_gb300.build`")
    lib = C.CDLL(path)
    for name, res, args in SIGNATURES:
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


class SPDError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


def check(rc: int, handle=None):
    if rc != SPD_OK:
        msg = load().spd_last_error(handle)
        raise SPDError(rc, msg.decode() if msg else "")
    return rc


# Thin same-name wrappers --------------------------------------------------------------
def spd_workspace_bytes(dims, pdm, cfg) -> int:
    out = C.c_size_t(0)
    check(load().spd_workspace_bytes(C.byref(dims), C.byref(pdm) if pdm is not None else None, C.byref(cfg),
                                     C.byref(out)))
    return out.value


def spd_create(dims, tw, pw, cfg, workspace_ptr: int, ws_bytes: int, stream_ptr: int):
    h = C.c_void_p(0)
    check(load().spd_create(C.byref(dims), C.byref(tw), C.byref(pw) if pw is not None else None, C.byref(cfg),
                            C.c_void_p(workspace_ptr), C.c_size_t(ws_bytes), C.c_void_p(stream_ptr), C.byref(h)))
    return h


def spd_prefill(h, prompt_ptr: int, prompt_len: int):
    check(load().spd_prefill(h, C.c_void_p(prompt_ptr), prompt_len), h)


def spd_step(h, n_steps: int, want_count: bool = True):
    c = C.c_int32(0)
    check(load().spd_step(h, n_steps, C.byref(c) if want_count else None), h)
    return c.value if want_count else None


def spd_generate(h, prompt_ptr: int, prompt_len: int, on_host: int, out_ptr: int):
    n = C.c_int32(0)
    st = spd_stats()
    check(load().spd_generate(h, C.c_void_p(prompt_ptr), prompt_len, on_host, C.c_void_p(out_ptr), C.byref(n),
                              C.byref(st)), h)
    return n.value, st


def spd_get_trace(h, max_recs: int, len_ptr: int = 0):
    recs = (spd_trace_rec * max(1, max_recs))()
    cnt = C.c_int32(0)
    check(load().spd_get_trace(h, recs, max_recs, C.c_void_p(len_ptr) if len_ptr else None, C.byref(cnt)), h)
    return recs, cnt.value


def spd_get_trace_view(h) -> spd_trace_view:
    v = spd_trace_view()
    check(load().spd_get_trace_view(h, C.byref(v)), h)
    return v


def spd_get_stats(h):
    st = spd_stats()
    check(load().spd_get_stats(h, C.byref(st)), h)
    return st


def spd_get_tokens(h, tokens_ptr: int, max_tokens: int) -> int:
    cnt = C.c_int32(0)
    check(load().spd_get_tokens(h, C.c_void_p(tokens_ptr), max_tokens, C.byref(cnt)), h)
    return cnt.value


def spd_read_buffer(h, which: int, index: int, offset: int, dst_ptr: int, nbytes: int):
    check(load().spd_read_buffer(h, which, index, offset, C.c_void_p(dst_ptr), nbytes), h)


def spd_kernel_timing(h):
    ms = C.c_double(0)
    n = C.c_int64(0)
    check(load().spd_kernel_timing(h, C.byref(ms), C.byref(n)), h)
    return ms.value, n.value


def check_op(rc: int):
    if rc != SPD_OK:
        msg = load().spd_ops_last_error()
        raise SPDError(rc, msg.decode() if msg else "")
    return rc


def spd_attention_scratch_bytes(Hq: int, Hkv: int, hd: int, seq_len: int) -> int:
    out = C.c_size_t(0)
    check_op(load().spd_attention_scratch_bytes(Hq, Hkv, hd, seq_len, C.byref(out)))
    return out.value


def spd_attention_decode(dtype: int, Hq: int, Hkv: int, hd: int, seq_len: int, q_ptr: int, k_ptr: int, v_ptr: int,
                         out_ptr: int, scratch_ptr: int, scratch_bytes: int, stream_ptr: int = 0):
    check_op(load().spd_attention_decode(dtype, Hq, Hkv, hd, seq_len, C.c_void_p(q_ptr), C.c_void_p(k_ptr),
                                         C.c_void_p(v_ptr), C.c_void_p(out_ptr), C.c_void_p(scratch_ptr),
                                         C.c_size_t(scratch_bytes), C.c_void_p(stream_ptr)))


def spd_attention_decode_noalloc(dtype: int, Hq: int, Hkv: int, hd: int, seq_len: int, q_ptr: int, k_ptr: int,
                                 v_ptr: int, out_ptr: int, stream_ptr: int = 0):
    check_op(load().spd_attention_decode_noalloc(dtype, Hq, Hkv, hd, seq_len, C.c_void_p(q_ptr), C.c_void_p(k_ptr),
                                                 C.c_void_p(v_ptr), C.c_void_p(out_ptr), C.c_void_p(stream_ptr)))


def spd_ops_last_error() -> str:
    m = load().spd_ops_last_error()
    return m.decode() if m else ""


def spd_reset(h):
    check(load().spd_reset(h), h)


def spd_destroy(h):
    load().spd_destroy(h)


def spd_last_error(h=None) -> str:
    m = load().spd_last_error(h)
    return m.decode() if m else ""
