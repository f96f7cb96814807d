"""ctypes binding of libeagle3.so: the C ABI of include/eagle3.h under the same names.

Argument marshalling only: device buffers are passed as integer addresses (e.g. a torch
tensor's ``data_ptr()``), host arrays as numpy int32 arrays, streams as integer handles.
Every computation happens in the CUDA library; if the library is missing this module
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libeagle3.so")

EAGLE3_OK = 0
EAGLE3_ERR_INVALID_ARG = -1
EAGLE3_ERR_CAPACITY = -2
EAGLE3_ERR_STATE = -3
EAGLE3_ERR_CUDA = -4
EAGLE3_ERR_DEVICE = -5
EAGLE3_ERR_UNSUPPORTED = -6
EAGLE3_SHRINK_GAMMA = 1
EAGLE3_DEV_BAD_TOKEN = 1
EAGLE3_DEV_BAD_PAGE = 2
EAGLE3_DEV_BAD_POSITION = 4
EAGLE3_DEV_BAD_LENGTH = 8
EAGLE3_DEV_TIMEOUT = 16

EXPORTED = (
    "eagle3_version", "eagle3_error_string", "eagle3_workspace_bytes", "eagle3_kv_row_bytes",
    "eagle3_resolve_rope_dims", "eagle3_config_from_json", "eagle3_selftest_bounded_wait",
    "eagle3_plan_gamma",
    "eagle3_init", "eagle3_destroy", "eagle3_encode", "eagle3_prefill", "eagle3_draft_chain",
    "eagle3_rewind", "eagle3_accept", "eagle3_verify_greedy", "eagle3_rebuild_after_verify",
    "eagle3_get_status",
    "eagle3_set_graph_mode", "eagle3_set_tc_min_items", "eagle3_set_tc_schedule", "eagle3_set_attention",
    "eagle3_launch_count", "eagle3_profile_begin",
    "eagle3_profile_end", "eagle3_profile_interval", "eagle3_lmhead_argmax_noalloc",
)


class Eagle3Error(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} ({code})")


class Config(ctypes.Structure):
    _fields_ = [("n_embd", ctypes.c_int), ("n_head", ctypes.c_int), ("n_head_kv", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("rope_dims", ctypes.c_int),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("n_ff", ctypes.c_int), ("draft_vocab", ctypes.c_int),
                ("target_vocab", ctypes.c_int), ("max_batch", ctypes.c_int),
                ("max_gamma", ctypes.c_int), ("max_cache_len", ctypes.c_int),
                ("page_size", ctypes.c_int), ("flags", ctypes.c_uint), ("kv_format", ctypes.c_int),
                ("weight_format", ctypes.c_int)]


EAGLE3_CKPT_NORM_BEFORE_RESIDUAL = 1
EAGLE3_W_BF16 = 0
EAGLE3_W_INT4_G128 = 1
EAGLE3_KV_BF16 = 0
EAGLE3_KV_Q8_0_Q5_1 = 1


WEIGHT_FIELDS = ("fc", "in_norm", "hidden_norm", "q", "k", "v", "o", "post_norm", "gate", "up",
                 "down", "final_norm", "lm_head", "embed", "d2t")


INT4_FIELDS = ("q_sz", "k_sz", "v_sz", "o_sz", "gate_sz", "up_sz", "down_sz", "lm_head_sz")


class Weights(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in WEIGHT_FIELDS + INT4_FIELDS]


class KV(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("num_pages", ctypes.c_int),
                ("max_pages_per_seq", ctypes.c_int), ("kv_len", ctypes.c_void_p)]


class Boundary(ctypes.Structure):
    _fields_ = [("g", ctypes.c_void_p), ("tok", ctypes.c_void_p)]


_lib = None


def load() -> ctypes.CDLL:
    """Load libeagle3.so (built by eagle_speculative_decode_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "eagle_speculative_decode_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, ci, cu = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint
    P = ctypes.POINTER
    sig = {
        "eagle3_version": (ci, []),
        "eagle3_error_string": (ctypes.c_char_p, [ci]),
        "eagle3_workspace_bytes": (ctypes.c_size_t, [P(Config)]),
        "eagle3_kv_row_bytes": (ci, [P(Config), P(ctypes.c_size_t), P(ctypes.c_size_t)]),
        "eagle3_resolve_rope_dims": (ci, [ci, ci, ci, ci, ctypes.c_float]),
        "eagle3_selftest_bounded_wait": (ci, [vp, vp, vp]),
        "eagle3_config_from_json": (ci, [ctypes.c_char_p, P(Config)]),
        "eagle3_plan_gamma": (ci, [ci, ci, ci, cu, P(ci)]),
        "eagle3_init": (ci, [P(Config), P(Weights), vp, ctypes.c_size_t, vp, P(vp)]),
        "eagle3_destroy": (ci, [vp]),
        "eagle3_encode": (ci, [vp, vp, ci, vp, vp]),
        "eagle3_prefill": (ci, [vp, ci, vp, ci, vp, vp, vp, P(KV), P(Boundary), vp]),
        "eagle3_draft_chain": (ci, [vp, ci, ci, cu, vp, P(KV), P(Boundary), vp, vp, vp, vp, vp, vp]),
        "eagle3_rewind": (ci, [vp, ci, P(KV), vp]),
        "eagle3_accept": (ci, [vp, ci, ci, vp, vp, vp, vp, vp, vp]),
        "eagle3_verify_greedy": (ci, [vp, ci, ci, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, vp]),
        "eagle3_rebuild_after_verify": (ci, [vp, ci, ci, vp, vp, vp, vp, P(KV), P(Boundary), vp]),
        "eagle3_get_status": (ci, [vp, P(ci)]),
        "eagle3_set_graph_mode": (ci, [vp, ci]),
        "eagle3_set_tc_min_items": (ci, [vp, ci]),
        "eagle3_set_tc_schedule": (ci, [vp, ci]),
        "eagle3_set_attention": (ci, [vp, ci]),
        "eagle3_launch_count": (ctypes.c_ulonglong, [vp]),
        "eagle3_profile_begin": (ci, [vp, ci]),
        "eagle3_profile_end": (ci, [vp, P(ci)]),
        "eagle3_profile_interval": (ci, [vp, ci, P(ci), P(ctypes.c_float)]),
        "eagle3_lmhead_argmax_noalloc": (ci, [vp, vp, vp, vp, ci, ci, ci, ci, ctypes.c_float,
                                              vp, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def error_string(code: int) -> str:
    return load().eagle3_error_string(int(code)).decode()


def _check(code: int, where: str) -> int:
    if code != EAGLE3_OK:
        raise Eagle3Error(code, where)
    return code


def _host_i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# -------------------------------------------------------------- thin wrappers

def eagle3_version() -> int:
    return load().eagle3_version()


def eagle3_workspace_bytes(cfg: Config) -> int:
    return int(load().eagle3_workspace_bytes(ctypes.byref(cfg)))


def eagle3_selftest_bounded_wait(device_status: int, device_result: int, stream: int = 0) -> None:
    _check(load().eagle3_selftest_bounded_wait(device_status, device_result, stream),
           "eagle3_selftest_bounded_wait")


def eagle3_resolve_rope_dims(head_dim: int, rotary_dim: int | None, factor: float | None) -> int:
    """Rotary width: explicit rotary_dim > partial_rotary_factor * head_dim > full width."""
    return int(load().eagle3_resolve_rope_dims(int(head_dim), 0 if rotary_dim is None else 1,
                                               0 if rotary_dim is None else int(rotary_dim),
                                               0 if factor is None else 1,
                                               0.0 if factor is None else float(factor)))


def eagle3_config_from_json(text: str, cfg: Config | None = None) -> Config:
    """Drafter shape and flags from a checkpoint config.json text, into cfg (or a new
    Config whose batch / cache fields are zero)."""
    cfg = cfg if cfg is not None else Config()
    _check(load().eagle3_config_from_json(text.encode(), ctypes.byref(cfg)), "eagle3_config_from_json")
    return cfg


def eagle3_kv_row_bytes(cfg: Config):
    """(K row bytes, V row bytes) of the paged pools for cfg's kv_format."""
    k, v = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().eagle3_kv_row_bytes(ctypes.byref(cfg), ctypes.byref(k), ctypes.byref(v)),
           "eagle3_kv_row_bytes")
    return int(k.value), int(v.value)


def eagle3_plan_gamma(kv_len: int, gamma: int, max_cache_len: int, flags: int = 0) -> int:
    """Returns gamma_eff; raises Eagle3Error (e.g. EAGLE3_ERR_CAPACITY)."""
    out = ctypes.c_int(0)
    _check(load().eagle3_plan_gamma(int(kv_len), int(gamma), int(max_cache_len), int(flags),
                                    ctypes.byref(out)), "eagle3_plan_gamma")
    return out.value


def eagle3_init(cfg: Config, weights: Weights, workspace: int, workspace_bytes: int,
                stream: int = 0) -> int:
    ctx = ctypes.c_void_p(0)
    _check(load().eagle3_init(ctypes.byref(cfg), ctypes.byref(weights), workspace,
                              workspace_bytes, stream, ctypes.byref(ctx)), "eagle3_init")
    return int(ctx.value)


def eagle3_destroy(ctx: int) -> None:
    _check(load().eagle3_destroy(ctx), "eagle3_destroy")


def eagle3_set_graph_mode(ctx: int, enabled: bool) -> None:
    _check(load().eagle3_set_graph_mode(ctx, 1 if enabled else 0), "eagle3_set_graph_mode")


def eagle3_set_tc_min_items(ctx: int, min_items: int) -> None:
    _check(load().eagle3_set_tc_min_items(ctx, min_items), "eagle3_set_tc_min_items")


def eagle3_set_tc_schedule(ctx: int, schedule: int) -> None:
    _check(load().eagle3_set_tc_schedule(ctx, schedule), "eagle3_set_tc_schedule")


def eagle3_set_attention(ctx: int, mode: int) -> None:
    _check(load().eagle3_set_attention(ctx, mode), "eagle3_set_attention")


def eagle3_encode(ctx: int, aux: int, M: int, g: int, stream: int = 0) -> None:
    _check(load().eagle3_encode(ctx, aux, int(M), g, stream), "eagle3_encode")


def eagle3_prefill(ctx: int, B: int, tokens: int, P_max: int, next_tok: int, prompt_len_host,
                   aux: int, kv: KV, bnd: Boundary, stream: int = 0) -> None:
    pl = _host_i32(prompt_len_host)
    _check(load().eagle3_prefill(ctx, int(B), tokens, int(P_max), next_tok,
                                 pl.ctypes.data_as(ctypes.c_void_p), aux, ctypes.byref(kv),
                                 ctypes.byref(bnd), stream), "eagle3_prefill")


def eagle3_draft_chain(ctx: int, B: int, gamma: int, flags: int, kv_len_host, kv: KV,
                       bnd: Boundary, draft_tok: int, draft_id: int | None = None,
                       gamma_eff: int | None = None, logits_dbg: int | None = None,
                       g_dbg: int | None = None, stream: int = 0) -> None:
    kl = _host_i32(kv_len_host)
    _check(load().eagle3_draft_chain(ctx, int(B), int(gamma), int(flags),
                                     kl.ctypes.data_as(ctypes.c_void_p), ctypes.byref(kv),
                                     ctypes.byref(bnd), draft_tok, draft_id, gamma_eff,
                                     logits_dbg, g_dbg, stream), "eagle3_draft_chain")


def eagle3_rewind(ctx: int, B: int, kv: KV, stream: int = 0) -> None:
    _check(load().eagle3_rewind(ctx, int(B), ctypes.byref(kv), stream), "eagle3_rewind")


def eagle3_accept(ctx: int, B: int, gamma: int, draft_tok: int, target_pred: int,
                  gamma_eff: int | None, n_acc: int, bonus: int, stream: int = 0) -> None:
    _check(load().eagle3_accept(ctx, int(B), int(gamma), draft_tok, target_pred, gamma_eff,
                                n_acc, bonus, stream), "eagle3_accept")


def eagle3_verify_greedy(ctx: int, B: int, gamma: int, target_lm_head: int, target_norm: int,
                         target_rms_eps: float, hidden: int, draft_tok: int, gamma_eff: int | None,
                         target_pred: int, n_acc: int, bonus: int, logits_dbg: int | None,
                         stream: int = 0) -> None:
    _check(load().eagle3_verify_greedy(ctx, int(B), int(gamma), target_lm_head, target_norm,
                                       float(target_rms_eps), hidden, draft_tok, gamma_eff,
                                       target_pred, n_acc, bonus, logits_dbg, stream),
           "eagle3_verify_greedy")


def eagle3_rebuild_after_verify(ctx: int, B: int, gamma: int, n_acc: int, draft_tok: int,
                                bonus: int, verify_aux: int, kv: KV, bnd: Boundary,
                                stream: int = 0) -> None:
    _check(load().eagle3_rebuild_after_verify(ctx, int(B), int(gamma), n_acc, draft_tok, bonus,
                                              verify_aux, ctypes.byref(kv), ctypes.byref(bnd),
                                              stream), "eagle3_rebuild_after_verify")


def eagle3_get_status(ctx: int) -> int:
    """Synchronises; returns the device status word (0 = clean) without raising."""
    s = ctypes.c_int(0)
    rc = load().eagle3_get_status(ctx, ctypes.byref(s))
    if rc not in (EAGLE3_OK, EAGLE3_ERR_DEVICE):
        raise Eagle3Error(rc, "eagle3_get_status")
    return s.value


def eagle3_launch_count(ctx: int) -> int:
    return int(load().eagle3_launch_count(ctx))


def eagle3_profile_begin(ctx: int, max_events: int) -> None:
    _check(load().eagle3_profile_begin(ctx, int(max_events)), "eagle3_profile_begin")


def eagle3_profile_end(ctx: int) -> list[tuple[int, float]]:
    """Stops recording; returns [(label, milliseconds)] for every recorded interval."""
    n = ctypes.c_int(0)
    _check(load().eagle3_profile_end(ctx, ctypes.byref(n)), "eagle3_profile_end")
    out = []
    lab, ms = ctypes.c_int(0), ctypes.c_float(0.0)
    for i in range(1, n.value):
        _check(load().eagle3_profile_interval(ctx, i, ctypes.byref(lab), ctypes.byref(ms)),
               "eagle3_profile_interval")
        out.append((lab.value, ms.value))
    return out


def eagle3_lmhead_argmax_noalloc(lm_head: int, final_norm: int, d2t: int, x: int, rows: int,
                                 n_embd: int, draft_vocab: int, target_vocab: int, rms_eps: float,
                                 draft_id: int | None, target_id: int, logits: int | None = None,
                                 stream: int = 0) -> None:
    _check(load().eagle3_lmhead_argmax_noalloc(lm_head, final_norm, d2t, x, int(rows), int(n_embd),
                                               int(draft_vocab), int(target_vocab), float(rms_eps),
                                               draft_id, target_id, logits, stream),
           "eagle3_lmhead_argmax_noalloc")
