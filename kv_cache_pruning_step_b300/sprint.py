"""Python binding of libsprint.so, the SPRINT C ABI (include/sprint.h).

Argument marshalling only: each function has the name of the C entry point
it calls, checks that tensors are contiguous CUDA tensors of the right
dtype, allocates outputs and the workspace with torch when the caller gives
none, passes raw pointers and the current CUDA stream, and raises
SprintError on a negative return code.  Every step of the computation runs
in the library's CUDA kernels; there is no other implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

# The release library next to this file, or the one SPRINT_LIBRARY names
# (the debug build, libsprint_debug.so).
LIB_PATH = os.environ.get("SPRINT_LIBRARY") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libsprint.so")

F32 = 0
BF16 = 1
UNMASK_ADAPTIVE = 0
UNMASK_FIXED = 1

STATUS_BAD_OFFSETS = 1
STATUS_KEPT_MISMATCH = 2
STATUS_TIMEOUT = 4
STATUS_BAD_INDEX = 8
STATUS_BAD_TEMPERATURE = 16
STATUS_DEBUG_CHECK = 32

# Every symbol include/sprint.h declares, with (restype, argtypes).
_P, _I, _Z, _F, _D = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_double
SIGNATURES = {
    "sprint_version": (_I, []),
    "sprint_strerror": (ctypes.c_char_p, [_I]),
    "sprint_kernel_launches": (ctypes.c_ulonglong, []),
    "sprint_debug_checks": (_I, []),
    "sprint_keep_count": (_I, [_I, _D]),
    "sprint_lmhead_workspace_bytes": (_Z, [_I, _I, _I, _I]),
    "sprint_lmhead_confidence": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P, _P]),
    "sprint_lmhead_confidence_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "sprint_score_prune_workspace_bytes": (_Z, [_I, _I]),
    "sprint_score_prune": (_I, [_P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _F, _D, _D, _P, _P,
                                _P, _P, _Z, _P, _P]),
    "sprint_key_norms": (_I, [_P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "sprint_select_kept_workspace_bytes": (_Z, [_I, _I]),
    "sprint_select_kept": (_I, [_P, _I, _P, _I, _P, _P, _F, _D, _D, _P, _P, _P, _P, _Z, _P,
                                _P]),
    "sprint_select_kept_pools_workspace_bytes": (_Z, [_I, _I, _I]),
    "sprint_select_kept_pools": (_I, [_P, _I, _P, _I, _P, _P, _I, _P, _F, _P, _P, _I, _P, _P,
                                      _Z, _P, _P]),
    "sprint_score_prune_pools_workspace_bytes": (_Z, [_I, _I, _I]),
    "sprint_score_prune_pools": (_I, [_P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _F, _P,
                                      _P, _I, _P, _P, _Z, _P, _P]),
    "sprint_compact_kv": (_I, [_P, _P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P]),
    "sprint_block_attn_workspace_bytes": (_Z, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "sprint_block_attn": (_I, [_P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P,
                               _P, _Z, _P, _P]),
    "sprint_block_attn_indexed": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _P, _P, _I, _I, _I,
                                       _I, _I, _I, _I, _P, _P, _Z, _P, _P]),
    "sprint_residual_hidden": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "sprint_prefix_attn": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "sprint_unmask": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P, _P]),
    "sprint_decode_steps": (_I, [_P, _P]),
}


class StepsArgs(ctypes.Structure):
    """Mirror of sprint_steps_args (include/sprint.h)."""
    _fields_ = [(n, ctypes.c_int) for n in ("S", "NL", "LB", "Hq", "Hkv", "d", "D", "vocab",
                                            "dtype", "T")] + [
        ("tau", ctypes.c_float), ("mode", ctypes.c_int),
        ("Kf", _P), ("Vf", _P), ("prefix_off", _P), ("max_rows", ctypes.c_int),
        ("total_rows", ctypes.c_int),
        ("Kp", _P), ("Vp", _P), ("kept_off", _P), ("max_kept", ctypes.c_int),
        ("total_kept", ctypes.c_int),
        ("W", _P), ("Q", _P), ("Kb", _P), ("Vb", _P), ("h", _P), ("theta", _P),
        ("O", _P), ("logits", _P), ("conf", _P), ("argmax", _P), ("mask", _P),
        ("tokens", _P), ("m_hist", _P), ("accepted", _P),
        ("ws_attn", _P), ("ws_attn_bytes", ctypes.c_size_t),
        ("ws_lm", _P), ("ws_lm_bytes", ctypes.c_size_t),
        ("status", _P), ("events", _P), ("kept_idx", _P),
        ("residual", ctypes.c_int), ("h_res", _P), ("step0_given", ctypes.c_int),
    ]


class SprintError(RuntimeError):
    pass


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -m kv_cache_pruning_step_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _check(rc: int, what: str):
    if rc != 0:
        raise SprintError(f"{what}: {lib.sprint_strerror(rc).decode()} (code {rc})")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise SprintError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise SprintError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise SprintError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise SprintError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr() if t.numel() else None


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ws(ws, nbytes, device):
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)
    return ws


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def sprint_version() -> int:
    return lib.sprint_version()


def sprint_strerror(code: int) -> str:
    return lib.sprint_strerror(code).decode()


def sprint_kernel_launches() -> int:
    return lib.sprint_kernel_launches()


def sprint_debug_checks() -> int:
    return lib.sprint_debug_checks()


def sprint_keep_count(n: int, r: float) -> int:
    return lib.sprint_keep_count(int(n), float(r))


def sprint_lmhead_workspace_bytes(M, D, V, dtype) -> int:
    return lib.sprint_lmhead_workspace_bytes(M, D, V, dtype)


def sprint_lmhead_confidence(h, W, temp=None, *, want_logits=False, conf=None, argmax=None,
                             logits=None, ws=None, status=None, stream=None, want_argmax=True):
    """c = top-1 softmax confidence and argmax token of every row of h @ W^T / temp.

    Returns (conf fp32 [M], argmax int32 [M] or None, logits [M][V] or None);
    want_argmax=False computes the confidence alone."""
    M, D = h.shape
    V = W.shape[0]
    dt = _dtype_code(h)
    dev = h.device
    conf = torch.empty(M, dtype=torch.float32, device=dev) if conf is None else conf
    if not want_argmax:
        argmax = None
    elif argmax is None:
        argmax = torch.empty(M, dtype=torch.int32, device=dev)
    if want_logits and logits is None:
        logits = torch.empty((M, V), dtype=h.dtype, device=dev)
    status = new_status(dev) if status is None else status
    nb = sprint_lmhead_workspace_bytes(M, D, V, dt)
    ws = _ws(ws, nb, dev)
    rc = lib.sprint_lmhead_confidence(
        _ptr(h, h.dtype, "h"), _ptr(W, h.dtype, "W"), _ptr(temp, torch.float32, "temp"),
        M, D, V, dt, _ptr(logits, h.dtype, "logits"), _ptr(conf, torch.float32, "conf"),
        _ptr(argmax, torch.int32, "argmax"), _ptr(ws), ws.numel(),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "sprint_lmhead_confidence")
    return conf, argmax, logits


def sprint_lmhead_confidence_noalloc(h, W, temp=None, *, want_logits=False, conf=None,
                                     argmax=None, logits=None, status=None, stream=None):
    """sprint_lmhead_confidence without a workspace: the library's fixed
    device scratch array holds the partials (see include/sprint.h for its
    size limit and for the sharing rules between calls)."""
    M, D = h.shape
    V = W.shape[0]
    dt = _dtype_code(h)
    dev = h.device
    conf = torch.empty(M, dtype=torch.float32, device=dev) if conf is None else conf
    argmax = torch.empty(M, dtype=torch.int32, device=dev) if argmax is None else argmax
    if want_logits and logits is None:
        logits = torch.empty((M, V), dtype=h.dtype, device=dev)
    status = new_status(dev) if status is None else status
    rc = lib.sprint_lmhead_confidence_noalloc(
        _ptr(h, h.dtype, "h"), _ptr(W, h.dtype, "W"), _ptr(temp, torch.float32, "temp"),
        M, D, V, dt, _ptr(logits, h.dtype, "logits"), _ptr(conf, torch.float32, "conf"),
        _ptr(argmax, torch.int32, "argmax"), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check(rc, "sprint_lmhead_confidence_noalloc")
    return conf, argmax, logits


def sprint_score_prune_workspace_bytes(S, total_rows) -> int:
    return lib.sprint_score_prune_workspace_bytes(S, total_rows)


def sprint_score_prune(K, prefix_off, total_rows, NL, Hkv, d, conf, modality, alpha,
                       r_text, r_img, kept_off, total_kept, *, kept_idx=None,
                       want_score=False, score=None, ws=None, status=None, stream=None):
    """Kept positions of every sequence (int32, local indices, ascending).

    Returns (kept_idx int32 [total_kept], score fp32 [total_rows] or None)."""
    S = prefix_off.numel() - 1
    dev = K.device
    dt = _dtype_code(K)
    kept_idx = (torch.empty(total_kept, dtype=torch.int32, device=dev)
                if kept_idx is None else kept_idx)
    if want_score and score is None:
        score = torch.empty(total_rows, dtype=torch.float32, device=dev)
    status = new_status(dev) if status is None else status
    ws = _ws(ws, sprint_score_prune_workspace_bytes(S, total_rows), dev)
    rc = lib.sprint_score_prune(
        _ptr(K, K.dtype, "K"), S, _ptr(prefix_off, torch.int32, "prefix_off"), int(total_rows),
        NL, Hkv, d, dt, _ptr(conf, torch.float32, "conf"),
        _ptr(modality, torch.uint8, "modality"), float(alpha), float(r_text), float(r_img),
        _ptr(kept_idx, torch.int32, "kept_idx"), _ptr(kept_off, torch.int32, "kept_off"),
        _ptr(score, torch.float32, "score"), _ptr(ws), ws.numel(),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "sprint_score_prune")
    return kept_idx, score


def sprint_key_norms(K, prefix_off, total_rows, NL, Hkv, d, *, u=None, status=None,
                     stream=None):
    """u fp32 [total_rows]: mean over layers of the L2 norm of every prefix
    position's keys (concatenated over the KV heads)."""
    S = prefix_off.numel() - 1
    dev = K.device
    u = torch.empty(total_rows, dtype=torch.float32, device=dev) if u is None else u
    status = new_status(dev) if status is None else status
    rc = lib.sprint_key_norms(
        _ptr(K, K.dtype, "K"), S, _ptr(prefix_off, torch.int32, "prefix_off"), int(total_rows),
        NL, Hkv, d, _dtype_code(K), _ptr(u, torch.float32, "u"),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "sprint_key_norms")
    return u


def sprint_select_kept_workspace_bytes(S, total_rows) -> int:
    return lib.sprint_select_kept_workspace_bytes(S, total_rows)


def sprint_select_kept(u, prefix_off, total_rows, conf, modality, alpha, r_text, r_img,
                       kept_off, total_kept, *, kept_idx=None, want_score=False, score=None,
                       ws=None, status=None, stream=None):
    """sprint_score_prune's scores and kept set from key norms u.  Returns
    (kept_idx int32 [total_kept], score fp32 [total_rows] or None)."""
    S = prefix_off.numel() - 1
    dev = u.device
    kept_idx = (torch.empty(total_kept, dtype=torch.int32, device=dev)
                if kept_idx is None else kept_idx)
    if want_score and score is None:
        score = torch.empty(total_rows, dtype=torch.float32, device=dev)
    status = new_status(dev) if status is None else status
    ws = _ws(ws, sprint_select_kept_workspace_bytes(S, total_rows), dev)
    rc = lib.sprint_select_kept(
        _ptr(u, torch.float32, "u"), S, _ptr(prefix_off, torch.int32, "prefix_off"),
        int(total_rows), _ptr(conf, torch.float32, "conf"),
        _ptr(modality, torch.uint8, "modality"), float(alpha), float(r_text), float(r_img),
        _ptr(kept_idx, torch.int32, "kept_idx"), _ptr(kept_off, torch.int32, "kept_off"),
        _ptr(score, torch.float32, "score"), _ptr(ws), ws.numel(),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "sprint_select_kept")
    return kept_idx, score


def sprint_select_kept_pools_workspace_bytes(S, total_rows, n_pools) -> int:
    return lib.sprint_select_kept_pools_workspace_bytes(S, total_rows, n_pools)


def sprint_select_kept_pools(u, prefix_off, total_rows, conf, pool, n_pools, keep, alpha,
                             kept_off, total_kept, *, kept_idx=None, want_score=False,
                             score=None, ws=None, status=None, stream=None):
    """sprint_score_prune_pools' scores and kept set from key norms u."""
    S = prefix_off.numel() - 1
    dev = u.device
    kept_idx = (torch.empty(total_kept, dtype=torch.int32, device=dev)
                if kept_idx is None else kept_idx)
    if want_score and score is None:
        score = torch.empty(total_rows, dtype=torch.float32, device=dev)
    status = new_status(dev) if status is None else status
    ws = _ws(ws, sprint_select_kept_pools_workspace_bytes(S, total_rows, n_pools), dev)
    rc = lib.sprint_select_kept_pools(
        _ptr(u, torch.float32, "u"), S, _ptr(prefix_off, torch.int32, "prefix_off"),
        int(total_rows), _ptr(conf, torch.float32, "conf"), _ptr(pool, torch.uint8, "pool"),
        int(n_pools), _ptr(keep, torch.int32, "keep"), float(alpha),
        _ptr(kept_idx, torch.int32, "kept_idx"), _ptr(kept_off, torch.int32, "kept_off"),
        int(total_kept), _ptr(score, torch.float32, "score"), _ptr(ws), ws.numel(),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "sprint_select_kept_pools")
    return kept_idx, score


def sprint_score_prune_pools_workspace_bytes(S, total_rows, n_pools) -> int:
    return lib.sprint_score_prune_pools_workspace_bytes(S, total_rows, n_pools)


def sprint_score_prune_pools(K, prefix_off, total_rows, NL, Hkv, d, conf, pool, n_pools, keep,
                             alpha, kept_off, total_kept, *, kept_idx=None, want_score=False,
                             score=None, ws=None, status=None, stream=None):
    """Kept positions with a keep count per pool (keep: int32 [S][n_pools]
    on the device).  Returns (kept_idx int32 [total_kept], score or None)."""
    S = prefix_off.numel() - 1
    dev = K.device
    dt = _dtype_code(K)
    kept_idx = (torch.empty(total_kept, dtype=torch.int32, device=dev)
                if kept_idx is None else kept_idx)
    if want_score and score is None:
        score = torch.empty(total_rows, dtype=torch.float32, device=dev)
    status = new_status(dev) if status is None else status
    ws = _ws(ws, sprint_score_prune_pools_workspace_bytes(S, total_rows, n_pools), dev)
    rc = lib.sprint_score_prune_pools(
        _ptr(K, K.dtype, "K"), S, _ptr(prefix_off, torch.int32, "prefix_off"), int(total_rows),
        NL, Hkv, d, dt, _ptr(conf, torch.float32, "conf"), _ptr(pool, torch.uint8, "pool"),
        int(n_pools), _ptr(keep, torch.int32, "keep"), float(alpha),
        _ptr(kept_idx, torch.int32, "kept_idx"), _ptr(kept_off, torch.int32, "kept_off"),
        int(total_kept), _ptr(score, torch.float32, "score"), _ptr(ws), ws.numel(),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "sprint_score_prune_pools")
    return kept_idx, score


def sprint_compact_kv(K, V, prefix_off, total_rows, NL, Hkv, d, kept_idx, kept_off,
                      total_kept, *, Kp=None, Vp=None, status=None, stream=None):
    """Gather of the kept rows: returns (Kp, Vp), flat [total_kept*NL*Hkv*d]."""
    S = prefix_off.numel() - 1
    dev = K.device
    n = int(total_kept) * NL * Hkv * d
    Kp = torch.empty(n, dtype=K.dtype, device=dev) if Kp is None else Kp
    Vp = torch.empty(n, dtype=K.dtype, device=dev) if Vp is None else Vp
    status = new_status(dev) if status is None else status
    rc = lib.sprint_compact_kv(
        _ptr(K, K.dtype, "K"), _ptr(V, K.dtype, "V"), S,
        _ptr(prefix_off, torch.int32, "prefix_off"), int(total_rows), NL, Hkv, d,
        _dtype_code(K), _ptr(kept_idx, torch.int32, "kept_idx"),
        _ptr(kept_off, torch.int32, "kept_off"), int(total_kept), _ptr(Kp, K.dtype, "Kp"),
        _ptr(Vp, K.dtype, "Vp"), _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "sprint_compact_kv")
    return Kp, Vp


def sprint_block_attn_workspace_bytes(S, NL, LB, Hq, Hkv, d, max_kv_rows, dtype) -> int:
    return lib.sprint_block_attn_workspace_bytes(S, NL, LB, Hq, Hkv, d, max_kv_rows, dtype)


def sprint_block_attn(Q, Kp, Vp, kv_off, max_kv_rows, total_kv_rows, Kb, Vb, *, O=None,
                      ws=None, status=None, stream=None):
    """Block attention; Q [S][NL][LB][Hq][d], Kb/Vb [S][NL][LB][Hkv][d]."""
    S, NL, LB, Hq, d = Q.shape
    Hkv = Kb.shape[3]
    dev = Q.device
    dt = _dtype_code(Q)
    O = torch.empty_like(Q) if O is None else O
    status = new_status(dev) if status is None else status
    ws = _ws(ws, sprint_block_attn_workspace_bytes(S, NL, LB, Hq, Hkv, d, int(max_kv_rows), dt),
             dev)
    rc = lib.sprint_block_attn(
        _ptr(Q, Q.dtype, "Q"), _ptr(Kp, Q.dtype, "Kp"), _ptr(Vp, Q.dtype, "Vp"),
        _ptr(kv_off, torch.int32, "kv_off"), int(max_kv_rows), int(total_kv_rows),
        _ptr(Kb, Q.dtype, "Kb"), _ptr(Vb, Q.dtype, "Vb"), S, NL, LB, Hq, Hkv, d, dt,
        _ptr(O, Q.dtype, "O"), _ptr(ws), ws.numel(), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check(rc, "sprint_block_attn")
    return O


def sprint_block_attn_indexed(Q, K, V, prefix_off, total_rows, kept_idx, kept_off, max_kept,
                              total_kept, Kb, Vb, *, O=None, ws=None, status=None, stream=None):
    """Block attention over the kept rows of the full cache K / V, read
    through kept_idx (no compacted copy); same output as sprint_compact_kv
    followed by sprint_block_attn."""
    S, NL, LB, Hq, d = Q.shape
    Hkv = Kb.shape[3]
    dev = Q.device
    dt = _dtype_code(Q)
    O = torch.empty_like(Q) if O is None else O
    status = new_status(dev) if status is None else status
    ws = _ws(ws, sprint_block_attn_workspace_bytes(S, NL, LB, Hq, Hkv, d, int(max_kept), dt),
             dev)
    rc = lib.sprint_block_attn_indexed(
        _ptr(Q, Q.dtype, "Q"), _ptr(K, Q.dtype, "K"), _ptr(V, Q.dtype, "V"),
        _ptr(prefix_off, torch.int32, "prefix_off"), int(total_rows),
        _ptr(kept_idx, torch.int32, "kept_idx"), _ptr(kept_off, torch.int32, "kept_off"),
        int(max_kept), int(total_kept), _ptr(Kb, Q.dtype, "Kb"), _ptr(Vb, Q.dtype, "Vb"),
        S, NL, LB, Hq, Hkv, d, dt, _ptr(O, Q.dtype, "O"), _ptr(ws), ws.numel(),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "sprint_block_attn_indexed")
    return O


def sprint_residual_hidden(h_in, O, *, h_out=None, stream=None):
    """h_out = h_in + O of the last layer, heads concatenated; O is
    [S][NL][LB][Hq][d], h_in [S*LB][Hq*d]."""
    S, NL, LB, Hq, d = O.shape
    h_out = torch.empty_like(h_in) if h_out is None else h_out
    rc = lib.sprint_residual_hidden(_ptr(h_in, O.dtype, "h_in"), _ptr(O, O.dtype, "O"), S, NL,
                                    LB, Hq, d, _dtype_code(O), _ptr(h_out, O.dtype, "h_out"),
                                    _stream(stream))
    _check(rc, "sprint_residual_hidden")
    return h_out


def sprint_prefix_attn(Qp, K, V, prefix_off, total_rows, NL, Hq, Hkv, d, *, Op=None,
                       status=None, stream=None):
    """The prefix's own attention at a block's first step: Op [NL][n_s][Hq][d]
    per sequence (concatenated like Qp), every position over every position
    of its sequence's prefix."""
    S = prefix_off.numel() - 1
    dev = Qp.device
    Op = torch.empty_like(Qp) if Op is None else Op
    status = new_status(dev) if status is None else status
    rc = lib.sprint_prefix_attn(
        _ptr(Qp, Qp.dtype, "Qp"), _ptr(K, Qp.dtype, "K"), _ptr(V, Qp.dtype, "V"),
        _ptr(prefix_off, torch.int32, "prefix_off"), int(total_rows), S, NL, Hq, Hkv, d,
        _dtype_code(Qp), _ptr(Op, Qp.dtype, "Op"), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check(rc, "sprint_prefix_attn")
    return Op


def sprint_unmask(conf, argmax, mask, tokens, t, T, tau, mode=UNMASK_ADAPTIVE, *, m_out=None,
                  accepted=None, status=None, stream=None):
    """One unmask step in place on mask/tokens ([S][LB]); returns (m_out, accepted)."""
    S, LB = mask.shape
    dev = mask.device
    m_out = torch.empty(S, dtype=torch.int32, device=dev) if m_out is None else m_out
    accepted = torch.empty((S, LB), dtype=torch.uint8, device=dev) if accepted is None else accepted
    status = new_status(dev) if status is None else status
    rc = lib.sprint_unmask(
        _ptr(conf, torch.float32, "conf"), _ptr(argmax, torch.int32, "argmax"),
        _ptr(mask, torch.uint8, "mask"), _ptr(tokens, torch.int32, "tokens"),
        _ptr(m_out, torch.int32, "m_out"), S, LB, int(t), int(T), float(tau), int(mode),
        _ptr(accepted, torch.uint8, "accepted"), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check(rc, "sprint_unmask")
    return m_out, accepted


def _ptr_array(tensors, dtype, name):
    arr = (ctypes.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = _ptr(t, dtype, f"{name}[{i}]") if t is not None else None
    return arr


def sprint_decode_steps(*, Q, Kb, Vb, h, theta, Kf, Vf, prefix_off, max_rows, total_rows,
                        Kp, Vp, kept_off, max_kept, total_kept, W, T, tau, mode, O, conf,
                        argmax, mask, tokens, m_hist, ws_attn, ws_lm, status, accepted=None,
                        logits=None, events=None, kept_idx=None, h_res=None,
                        step0_given=False, stream=None):
    """Every denoising step of one block in one call (see include/sprint.h).

    Q, Kb, Vb: lists of T tensors [S][NL][LB][*][d]; h: list of T [S*LB][D];
    theta: list of T [S*LB] fp32 or None.  m_hist: int32 [T][S] (out);
    events: list of 6*T torch.cuda.Event (or None entries) or None; kept_idx: steps t >= 1
    read the kept rows of Kf / Vf through it (Kp / Vp unused); h_res: the
    LM head reads h_res = h[t] + O of the last layer (written by the
    attention)."""
    S, NL, LB, Hq, d = Q[0].shape
    Hkv = Kb[0].shape[3]
    dt = _dtype_code(Q[0])
    a = StepsArgs()
    a.S, a.NL, a.LB, a.Hq, a.Hkv, a.d = S, NL, LB, Hq, Hkv, d
    a.D, a.vocab, a.dtype, a.T = W.shape[1], W.shape[0], dt, int(T)
    a.tau, a.mode = float(tau), int(mode)
    a.Kf, a.Vf = _ptr(Kf, Q[0].dtype, "Kf"), _ptr(Vf, Q[0].dtype, "Vf")
    a.prefix_off = _ptr(prefix_off, torch.int32, "prefix_off")
    a.max_rows, a.total_rows = int(max_rows), int(total_rows)
    a.Kp, a.Vp = _ptr(Kp, Q[0].dtype, "Kp"), _ptr(Vp, Q[0].dtype, "Vp")
    a.kept_off = _ptr(kept_off, torch.int32, "kept_off")
    a.max_kept, a.total_kept = int(max_kept), int(total_kept)
    a.W = _ptr(W, Q[0].dtype, "W")
    keep = [_ptr_array(Q, Q[0].dtype, "Q"), _ptr_array(Kb, Q[0].dtype, "Kb"),
            _ptr_array(Vb, Q[0].dtype, "Vb"), _ptr_array(h, Q[0].dtype, "h"),
            _ptr_array(theta if theta is not None else [None] * T, torch.float32, "theta")]
    a.Q, a.Kb, a.Vb, a.h, a.theta = [ctypes.cast(x, ctypes.c_void_p) for x in keep]
    a.O, a.logits = _ptr(O, Q[0].dtype, "O"), _ptr(logits, Q[0].dtype, "logits")
    a.conf, a.argmax = _ptr(conf, torch.float32, "conf"), _ptr(argmax, torch.int32, "argmax")
    a.mask, a.tokens = _ptr(mask, torch.uint8, "mask"), _ptr(tokens, torch.int32, "tokens")
    a.m_hist = _ptr(m_hist, torch.int32, "m_hist")
    a.accepted = _ptr(accepted, torch.uint8, "accepted")
    a.ws_attn, a.ws_attn_bytes = _ptr(ws_attn), ws_attn.numel()
    a.ws_lm, a.ws_lm_bytes = _ptr(ws_lm), ws_lm.numel()
    a.status = _ptr(status, torch.int32, "status")
    a.kept_idx = _ptr(kept_idx, torch.int32, "kept_idx")
    a.residual = 1 if h_res is not None else 0
    a.h_res = _ptr(h_res, Q[0].dtype, "h_res")
    a.step0_given = 1 if step0_given else 0
    ev = None
    if events is not None:
        ev = (ctypes.c_void_p * len(events))(*[e.cuda_event if e is not None else None
                                                for e in events])
        a.events = ctypes.cast(ev, ctypes.c_void_p)
    rc = lib.sprint_decode_steps(ctypes.byref(a), _stream(stream))
    _check(rc, "sprint_decode_steps")
    del keep, ev
