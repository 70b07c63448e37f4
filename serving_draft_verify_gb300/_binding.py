"""ctypes binding of libdspark.so: argument marshalling only.

Every function here has the name of the C entry point it calls and takes torch
tensors on the GPU; it checks shapes and dtypes, passes data pointers and the
current CUDA stream, and raises DSparkError on a non-OK status.  All compute
runs in the library's CUDA kernels -- there is no fallback of any kind: if the
library is missing, every call raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdspark.so")

DSPARK_OK = 0
DSPARK_F32 = 0
DSPARK_BF16 = 1
MAX_GAMMA = 32

_c_int, _c_i64, _c_u64, _c_size, _c_float = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                                            ctypes.c_size_t, ctypes.c_float)
_p = ctypes.c_void_p

_SIGNATURES = {
    "dspark_status_string": (ctypes.c_char_p, [_c_int]),
    "dspark_workspace_status": (_c_int, [_p, _p]),
    "dspark_set_l2_residency": (_c_int, [_c_size]),
    "dspark_draft_block_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "dspark_draft_block": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _p, _p, _p, _p, _p,
                                    _c_float, _p, _c_float, _c_u64, _p, _p, _p, _p, _p, _p, _c_size, _p]),
    "dspark_draft_block_noalloc": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _p, _p, _p, _p, _p,
                                            _c_float, _p, _c_float, _c_u64, _p, _p, _p, _p, _p, _p]),
    "dspark_schedule_prefix_workspace_size": (_c_size, [_c_int, _c_int]),
    "dspark_schedule_prefix": (_c_int, [_c_int, _c_int, _p, _p, _p, _p, _p, _p, _c_size, _p]),
    "dspark_verify_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "dspark_verify": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                               _c_float, _c_u64, _p, _p, _p, _c_size, _p]),
    "dspark_accept_rate_tv_workspace_size": (_c_size, [_c_i64, _c_int]),
    "dspark_accept_rate_tv": (_c_int, [_c_i64, _c_int, _c_int, _p, _p, _p, _p, _c_size, _p]),
    "dspark_training_loss_workspace_size": (_c_size, [_c_i64, _c_int]),
    "dspark_training_loss": (_c_int, [_c_i64, _c_int, _c_int, _p, _p, _p, _p, _p, _c_float, _c_float, _c_float,
                                      _p, _p, _p, _p, _p, _c_size, _p]),
    "dspark_decode_rounds_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "dspark_decode_rounds": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _p, _p, _p,
                                      _p, _p, _p, _c_float, _p, _p, _c_float, _c_u64, _p, _p, _p, _p, _p, _c_size,
                                      _p]),
    "dspark_draft_block_ex_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "dspark_draft_block_ex": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _p, _p, _p, _p, _p,
                                       _c_float, _p, _c_float, _c_u64, _p, _p, _p, _p, _p, _p, _p, _c_size, _p]),
    "dspark_verify_ex": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                                  _c_float, _c_u64, _p, _p, _p, _p, _c_size, _p]),
    "dspark_debug_draft_logits": (_c_int, [_c_int, _c_int, _c_int, _p, _p, _p, _p, _p, _p, _c_size, _p]),
    "dspark_debug_enable_phase_timing": (_c_int, [_c_int]),
    "dspark_debug_phase_times": (_c_int, [_p, _c_int]),
    "dspark_debug_force_phase_launches": (_c_int, [_c_int]),
    "dspark_debug_set_draft_path": (_c_int, [_c_int]),
    "dspark_debug_staged_bytes": (ctypes.c_uint64, []),
    "dspark_debug_bounded_wait": (_c_int, [_p, _c_size, ctypes.c_uint64, _p]),
    "dspark_debug_exp_draws": (_c_int, [_p, _p, _c_i64, _p]),
    "dspark_debug_philox_rows": (_c_int, [_c_u64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                          ctypes.c_uint32, _c_i64, _p, _p]),
}

_lib = None


class DSparkError(RuntimeError):
    def __init__(self, name, status):
        self.status = status
        super().__init__(f"{name} failed: {status_string(status) if _lib else status}")


def load():
    """Load libdspark.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols():
    return sorted(_SIGNATURES)


def status_string(status):
    return load().dspark_status_string(int(status)).decode()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(*ts):
    dts = {t.dtype for t in ts}
    if len(dts) != 1:
        raise TypeError(f"float inputs must share one dtype, got {dts}")
    dt = dts.pop()
    if dt == torch.bfloat16:
        return DSPARK_BF16
    if dt == torch.float32:
        return DSPARK_F32
    raise TypeError(f"unsupported dtype {dt}")


def _check(name, status):
    if status != DSPARK_OK:
        raise DSparkError(name, status)


def _need(t, shape, dtype=None, name="tensor", host_ok=False):
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _workspace(nbytes, device, workspace):
    if workspace is None:
        return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError("workspace too small")
    return workspace


def _nbytes(t):
    return t.numel() * t.element_size()


def workspace_status(workspace, stream=None):
    """Device status code left at the head of `workspace` (synchronises)."""
    return load().dspark_workspace_status(_ptr(workspace), _stream(stream))


def dspark_set_l2_residency(nbytes):
    """Opt-in: keep W2 (the Markov weight streamed every draft position) in L2 by a
    persisting access-policy window on the draft and residual launches; sets the
    current context's persisting-L2 limit to min(nbytes, the device maximum).
    0 turns it off and restores the previous limit.  Results are unchanged."""
    _check("dspark_set_l2_residency", load().dspark_set_l2_residency(int(nbytes)))


# ----------------------------------------------------------------- calls ---
def dspark_accept_rate_tv(d, t, c_star=None, workspace=None, stream=None):
    """c*[row] = 1 - 1/2 ||softmax(d[row]) - softmax(t[row])||_1 (float32 [rows])."""
    lib = load()
    rows, V = d.shape
    _need(d, (rows, V), name="d")
    _need(t, (rows, V), d.dtype, name="t")
    dt = _dtype_code(d, t)
    if c_star is None:
        c_star = torch.empty(rows, dtype=torch.float32, device=d.device)
    _need(c_star, (rows,), torch.float32, name="c_star")
    ws = _workspace(lib.dspark_accept_rate_tv_workspace_size(rows, V), d.device, workspace)
    _check("dspark_accept_rate_tv",
           lib.dspark_accept_rate_tv(rows, V, dt, _ptr(d), _ptr(t), _ptr(c_star), _ptr(ws), _nbytes(ws),
                                     _stream(stream)))
    return c_star


def dspark_training_loss(d, t, target, conf_logit, omega, alpha_ce=0.1, alpha_l1=0.9, alpha_conf=1.0,
                         grad=True, out=None, workspace=None, stream=None):
    """Joint loss; returns dict row [rows, 4] (ce, c*, bce, row), loss [1] and,
    with grad=True, grad_d [rows, V] (d's dtype) and grad_conf [rows]."""
    lib = load()
    rows, V = d.shape
    _need(d, (rows, V), name="d")
    _need(t, (rows, V), d.dtype, name="t")
    _need(target, (rows,), torch.int32, name="target")
    _need(conf_logit, (rows,), torch.float32, name="conf_logit")
    _need(omega, (rows,), torch.float32, name="omega")
    dt = _dtype_code(d, t)
    dev = d.device
    if out is None:
        out = dict(row=torch.empty((rows, 4), dtype=torch.float32, device=dev),
                   loss=torch.empty(1, dtype=torch.float32, device=dev))
        if grad:
            out["grad_d"] = torch.empty((rows, V), dtype=d.dtype, device=dev)
            out["grad_conf"] = torch.empty(rows, dtype=torch.float32, device=dev)
    _need(out["row"], (rows, 4), torch.float32, name="row")
    _need(out["loss"], (1,), torch.float32, name="loss")
    gd, gc = out.get("grad_d"), out.get("grad_conf")
    if gd is not None:
        _need(gd, (rows, V), d.dtype, name="grad_d")
    if gc is not None:
        _need(gc, (rows,), torch.float32, name="grad_conf")
    ws = _workspace(lib.dspark_training_loss_workspace_size(rows, V), dev, workspace)
    _check("dspark_training_loss",
           lib.dspark_training_loss(rows, V, dt, _ptr(d), _ptr(t), _ptr(target), _ptr(conf_logit), _ptr(omega),
                                    float(alpha_ce), float(alpha_l1), float(alpha_conf), _ptr(out["row"]),
                                    _ptr(out["loss"]), _ptr(gd), _ptr(gc), _ptr(ws), _nbytes(ws),
                                    _stream(stream)))
    return out


class _RoundTrace(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "lse_d", "logp_d", "c", "a", "ell", "n_accept", "next_token")]


def dspark_decode_rounds(U, h, t, W1, W2, w, bias, sps, anchor, rounds, temperature, seed, trace=False, out=None,
                         workspace=None, stream=None):
    """`rounds` draft -> schedule -> verify rounds over the pool U [P, B, gamma, V],
    h [P, B, gamma, H], t [P, B, gamma+1, V]; `anchor` [B] int32 is updated in place
    to the last emitted tokens.  Returns dict tokens [rounds, B, gamma+1],
    n_emitted [rounds, B], stats [rounds, 2] (E[tau], realised tokens per request)
    and, with trace=True, the per-round x, lse_d, logp_d, c, a, ell, n_accept,
    next_token."""
    lib = load()
    P, B, G, V = U.shape
    H = h.shape[-1]
    r = W1.shape[-1]
    _need(U, (P, B, G, V), name="U")
    _need(h, (P, B, G, H), U.dtype, name="h")
    _need(t, (P, B, G + 1, V), U.dtype, name="t", host_ok=True)   # pinned host: rows read in place
    _need(W1, (V, r), U.dtype, name="W1")
    _need(W2, (V, r), U.dtype, name="W2")
    _need(w, (H + r,), U.dtype, name="w")
    _need(sps, (B * (G + 1) + 1,), torch.float64, name="sps", host_ok=True)
    _need(anchor, (B,), torch.int32, name="anchor")
    dt = _dtype_code(U, h, t, W1, W2, w)
    dev = U.device
    if out is None:
        out = dict(tokens=torch.empty((rounds, B, G + 1), dtype=torch.int32, device=dev),
                   n_emitted=torch.empty((rounds, B), dtype=torch.int32, device=dev),
                   stats=torch.empty((rounds, 2), dtype=torch.float64, device=dev))
        if trace:
            for k in ("x",):
                out[k] = torch.empty((rounds, B, G), dtype=torch.int32, device=dev)
            for k in ("lse_d", "logp_d", "c", "a"):
                out[k] = torch.empty((rounds, B, G), dtype=torch.float32, device=dev)
            for k in ("ell", "n_accept", "next_token"):
                out[k] = torch.empty((rounds, B), dtype=torch.int32, device=dev)
    _need(out["tokens"], (rounds, B, G + 1), torch.int32, name="tokens")
    _need(out["n_emitted"], (rounds, B), torch.int32, name="n_emitted")
    _need(out["stats"], (rounds, 2), torch.float64, name="stats")
    tr = None
    if any(n in out for n, _ in _RoundTrace._fields_):
        for n, _ in _RoundTrace._fields_:
            if n in out:
                _need(out[n], (rounds, B, G) if n in ("x", "lse_d", "logp_d", "c", "a") else (rounds, B),
                      torch.int32 if n in ("x", "ell", "n_accept", "next_token") else torch.float32, name=n)
        tr = _RoundTrace(*[out[n].data_ptr() if n in out else None for n, _ in _RoundTrace._fields_])
    ws = _workspace(lib.dspark_decode_rounds_workspace_size(B, G, V, r), dev, workspace)
    _check("dspark_decode_rounds",
           lib.dspark_decode_rounds(rounds, P, B, G, V, H, r, dt, _ptr(U), _ptr(h), _ptr(t), _ptr(W1), _ptr(W2),
                                    _ptr(w), float(bias), _ptr(sps), _ptr(anchor), float(temperature),
                                    int(seed) & ((1 << 64) - 1), _ptr(out["tokens"]), _ptr(out["n_emitted"]),
                                    _ptr(out["stats"]), ctypes.addressof(tr) if tr is not None else None, _ptr(ws),
                                    _nbytes(ws), _stream(stream)))
    return out


def dspark_draft_block(U, h, W1, W2, w, bias, x0, temperature, seed, out=None, workspace=None,
                       stream=None):
    """Draft block; returns dict x, lse_d, logp_d, c, a (each [B, gamma]).  U, h and x0 may
    be pinned host tensors: the kernels then read them over the host link (each byte once)."""
    lib = load()
    B, G, V = U.shape
    H = h.shape[-1]
    r = W1.shape[-1]
    _need(U, (B, G, V), name="U", host_ok=True)
    _need(h, (B, G, H), U.dtype, name="h", host_ok=True)
    _need(W1, (V, r), U.dtype, name="W1")
    _need(W2, (V, r), U.dtype, name="W2")
    _need(w, (H + r,), U.dtype, name="w")
    _need(x0, (B,), torch.int32, name="x0", host_ok=True)
    dt = _dtype_code(U, h, W1, W2, w)
    dev = W1.device
    if out is None:
        out = dict(x=torch.empty((B, G), dtype=torch.int32, device=dev),
                   **{k: torch.empty((B, G), dtype=torch.float32, device=dev)
                      for k in ("lse_d", "logp_d", "c", "a")})
    ws = _workspace(lib.dspark_draft_block_workspace_size(B, G, V, r), dev, workspace)
    _check("dspark_draft_block",
           lib.dspark_draft_block(B, G, V, H, r, dt, _ptr(U), _ptr(h), _ptr(W1), _ptr(W2), _ptr(w),
                                  float(bias), _ptr(x0), float(temperature), int(seed) & (2**64 - 1),
                                  _ptr(out["x"]), _ptr(out["lse_d"]), _ptr(out["logp_d"]),
                                  _ptr(out["c"]), _ptr(out["a"]), _ptr(ws), _nbytes(ws), _stream(stream)))
    return out


HEAD_MARKOV, HEAD_GATED, HEAD_RNN = 0, 1, 2


class _Head(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("Wg", ctypes.c_void_p), ("Wc", ctypes.c_void_p), ("E", ctypes.c_void_p)]


def _head_struct(head, B, G, H, r, dtype, dev):
    """ctypes head descriptor from a dict {kind, Wg, Wc, E}; allocates E if absent."""
    kind = int(head["kind"])
    if kind == HEAD_MARKOV:
        return _Head(kind, None, None, None), None
    ldw = H + r if kind == HEAD_GATED else 2 * r + H
    _need(head["Wg"], (r, ldw), dtype, name="Wg")
    if kind == HEAD_RNN:
        _need(head["Wc"], (r, ldw), dtype, name="Wc")
    E = head.get("E")
    if E is None:
        E = torch.empty((B, G, r), dtype=dtype, device=dev)
    _need(E, (B, G, r), dtype, name="E")
    Wc = head.get("Wc")
    return _Head(kind, head["Wg"].data_ptr(), Wc.data_ptr() if Wc is not None else None, E.data_ptr()), E


def dspark_draft_block_ex(U, h, W1, W2, w, bias, x0, temperature, seed, head, out=None, workspace=None,
                          stream=None):
    """Draft block with a sequential head: head = dict(kind=HEAD_GATED or HEAD_RNN,
    Wg=[r, H+r] or [r, 2r+H], Wc=[r, 2r+H] (RNN), E=[B, gamma, r] (optional)).
    Returns dict x, lse_d, logp_d, c, a and E (the rank-r rows the bias used)."""
    lib = load()
    B, G, V = U.shape
    H = h.shape[-1]
    r = W1.shape[-1]
    _need(U, (B, G, V), name="U")
    _need(h, (B, G, H), U.dtype, name="h")
    _need(W1, (V, r), U.dtype, name="W1")
    _need(W2, (V, r), U.dtype, name="W2")
    _need(w, (H + r,), U.dtype, name="w")
    _need(x0, (B,), torch.int32, name="x0")
    dt = _dtype_code(U, h, W1, W2, w)
    dev = U.device
    hs, E = _head_struct(head, B, G, H, r, U.dtype, dev)
    if out is None:
        out = dict(x=torch.empty((B, G), dtype=torch.int32, device=dev),
                   **{k: torch.empty((B, G), dtype=torch.float32, device=dev)
                      for k in ("lse_d", "logp_d", "c", "a")})
    ws = _workspace(lib.dspark_draft_block_ex_workspace_size(B, G, V, r, int(head["kind"])), dev, workspace)
    _check("dspark_draft_block_ex",
           lib.dspark_draft_block_ex(B, G, V, H, r, dt, _ptr(U), _ptr(h), _ptr(W1), _ptr(W2), _ptr(w),
                                     float(bias), _ptr(x0), float(temperature), int(seed) & (2**64 - 1),
                                     ctypes.addressof(hs), _ptr(out["x"]), _ptr(out["lse_d"]), _ptr(out["logp_d"]),
                                     _ptr(out["c"]), _ptr(out["a"]), _ptr(ws), _nbytes(ws), _stream(stream)))
    out["E"] = E
    return out


def dspark_draft_block_noalloc(U, h, W1, W2, w, bias, x0, temperature, seed, out, stream=None):
    """dspark_draft_block with the library's fixed internal scratch (no workspace);
    for hosts that forbid device allocation.  `out` must hold preallocated
    x [B, gamma] int32 and lse_d, logp_d, c, a [B, gamma] float32."""
    lib = load()
    B, G, V = U.shape
    H = h.shape[-1]
    r = W1.shape[-1]
    _need(U, (B, G, V), name="U", host_ok=True)
    _need(h, (B, G, H), U.dtype, name="h", host_ok=True)
    _need(W1, (V, r), U.dtype, name="W1")
    _need(W2, (V, r), U.dtype, name="W2")
    _need(w, (H + r,), U.dtype, name="w")
    _need(x0, (B,), torch.int32, name="x0", host_ok=True)
    _need(out["x"], (B, G), torch.int32, name="x")
    for k in ("lse_d", "logp_d", "c", "a"):
        _need(out[k], (B, G), torch.float32, name=k)
    dt = _dtype_code(U, h, W1, W2, w)
    _check("dspark_draft_block_noalloc",
           lib.dspark_draft_block_noalloc(B, G, V, H, r, dt, _ptr(U), _ptr(h), _ptr(W1), _ptr(W2), _ptr(w),
                                          float(bias), _ptr(x0), float(temperature), int(seed) & (2**64 - 1),
                                          _ptr(out["x"]), _ptr(out["lse_d"]), _ptr(out["logp_d"]), _ptr(out["c"]),
                                          _ptr(out["a"]), _stream(stream)))
    return out


def dspark_schedule_prefix(a, sps, out=None, workspace=None, stream=None):
    """Algorithm 1; returns dict ell [B] int32, n_sched [1] int32, theta [1] float64."""
    lib = load()
    B, G = a.shape
    _need(a, (B, G), torch.float32, name="a")
    _need(sps, (B * (G + 1) + 1,), torch.float64, name="sps", host_ok=True)
    dev = a.device
    if out is None:
        out = dict(ell=torch.empty(B, dtype=torch.int32, device=dev),
                   n_sched=torch.empty(1, dtype=torch.int32, device=dev),
                   theta=torch.empty(1, dtype=torch.float64, device=dev))
    ws = _workspace(lib.dspark_schedule_prefix_workspace_size(B, G), dev, workspace)
    _check("dspark_schedule_prefix",
           lib.dspark_schedule_prefix(B, G, _ptr(a), _ptr(sps), _ptr(out["ell"]), _ptr(out["n_sched"]),
                                      _ptr(out["theta"]), _ptr(ws), _nbytes(ws), _stream(stream)))
    return out


def dspark_verify(t_logits, U, W1, W2, x0, x, lse_d, logp_d, ell, temperature, seed, out=None,
                  workspace=None, stream=None):
    """Verification; returns dict n_accept [B], next_token [B] (int32).  t_logits, U and x0
    may be pinned host tensors: the kernels then read the rows verification needs (the
    scheduled prefix and its bonus row; U rows of rejected requests only) over the host
    link, and no others."""
    lib = load()
    B, G, V = U.shape
    r = W1.shape[-1]
    _need(t_logits, (B, G + 1, V), U.dtype, name="t_logits", host_ok=True)
    _need(U, (B, G, V), name="U", host_ok=True)
    _need(W1, (V, r), U.dtype, name="W1")
    _need(W2, (V, r), U.dtype, name="W2")
    _need(x0, (B,), torch.int32, name="x0", host_ok=True)
    _need(x, (B, G), torch.int32, name="x")
    _need(lse_d, (B, G), torch.float32, name="lse_d")
    _need(logp_d, (B, G), torch.float32, name="logp_d")
    _need(ell, (B,), torch.int32, name="ell")
    dt = _dtype_code(t_logits, U, W1, W2)
    dev = W1.device
    if out is None:
        out = dict(n_accept=torch.empty(B, dtype=torch.int32, device=dev),
                   next_token=torch.empty(B, dtype=torch.int32, device=dev))
    ws = _workspace(lib.dspark_verify_workspace_size(B, G, V, r), dev, workspace)
    _check("dspark_verify",
           lib.dspark_verify(B, G, V, r, dt, _ptr(t_logits), _ptr(U), _ptr(W1), _ptr(W2), _ptr(x0),
                             _ptr(x), _ptr(lse_d), _ptr(logp_d), _ptr(ell), float(temperature),
                             int(seed) & (2**64 - 1), _ptr(out["n_accept"]), _ptr(out["next_token"]),
                             _ptr(ws), _nbytes(ws), _stream(stream)))
    return out


def dspark_debug_draft_logits(U_k, W1, W2, prev, z=None, workspace=None, stream=None):
    """Test hook: z = U_k + W2 . W1[prev] through the tensor-core draft path."""
    lib = load()
    B, V = U_k.shape
    r = W1.shape[-1]
    _need(W1, (V, r), U_k.dtype, name="W1")
    _need(W2, (V, r), U_k.dtype, name="W2")
    _need(prev, (B,), torch.int32, name="prev")
    if z is None:
        z = torch.empty((B, V), dtype=torch.float32, device=U_k.device)
    ws = _workspace(lib.dspark_draft_block_workspace_size(B, 1, V, r), U_k.device, workspace)
    _check("dspark_debug_draft_logits",
           lib.dspark_debug_draft_logits(B, V, r, _ptr(U_k), _ptr(W1), _ptr(W2), _ptr(prev), _ptr(z), _ptr(ws),
                                         _nbytes(ws), _stream(stream)))
    return z, ws


def phase_timing(enable):
    """Measurement hook: record CUDA events around every draft phase launch."""
    _check("dspark_debug_enable_phase_timing", load().dspark_debug_enable_phase_timing(1 if enable else 0))


def staged_bytes():
    """Measurement hook: bytes of host inputs the library has staged to the device by
    copy engine so far in this process."""
    return int(load().dspark_debug_staged_bytes())


def force_phase_launches(enable):
    """Test hook: the tensor-core draft path launches per position instead of
    its single cooperative launch."""
    _check("dspark_debug_force_phase_launches", load().dspark_debug_force_phase_launches(1 if enable else 0))


def set_draft_path(mode):
    """Test hook: 0 chooses the draft path by batch size, 1 always takes the
    tcgen05 engine, 2 the small-batch GEMV path wherever it applies (B <= 16)."""
    _check("dspark_debug_set_draft_path", load().dspark_debug_set_draft_path(int(mode)))


def bounded_wait(limit_ns, workspace=None, stream=None):
    """Test hook: a wait that nothing ends, bounded by limit_ns; returns the workspace."""
    lib = load()
    ws = _workspace(lib.dspark_draft_block_workspace_size(1, 1, 1, 8), torch.device("cuda"), workspace)
    _check("dspark_debug_bounded_wait", lib.dspark_debug_bounded_wait(_ptr(ws), _nbytes(ws), int(limit_ns),
                                                                      _stream(stream)))
    return ws


def exp_draws(words, stream=None):
    """E = -ln u of the sampler's noise for uint32 words (an int32 / int64 CUDA tensor
    holding the 32-bit patterns), computed by the library's device routine."""
    w = words.to(torch.int32).contiguous()
    E = torch.empty(w.shape, dtype=torch.float32, device=w.device)
    _check("dspark_debug_exp_draws", load().dspark_debug_exp_draws(_ptr(w), _ptr(E), w.numel(), _stream(stream)))
    return E


def philox_rows(seed, k, b, stream_id, q0, n, device="cuda", stream=None):
    """[n, 4] words of Philox4x32-10 at counters (q0 + i, k, b, stream_id) (int64 tensor
    of the unsigned 32-bit values), computed by the library's per-row device routine."""
    out = torch.empty((int(n), 4), dtype=torch.int32, device=device)
    _check("dspark_debug_philox_rows",
           load().dspark_debug_philox_rows(int(seed) & (2 ** 64 - 1), int(k), int(b), int(stream_id), int(q0),
                                           int(n), _ptr(out), _stream(stream)))
    return out.to(torch.int64) & 0xFFFFFFFF


def phase_times():
    """Durations (ms) of the phase launches of the most recent draft call."""
    buf = (ctypes.c_float * 64)()
    n = load().dspark_debug_phase_times(ctypes.cast(buf, ctypes.c_void_p), 64)
    return [buf[i] for i in range(n)]


def dspark_verify_ex(t_logits, U, W1, W2, x0, x, lse_d, logp_d, ell, temperature, seed, head, out=None,
                     workspace=None, stream=None):
    """Verification of a draft made with a sequential head: head = dict(kind, E)
    where E [B, gamma, r] holds the rows the draft's bias used (t_logits as for dspark_verify)."""
    lib = load()
    B, G, V = U.shape
    r = W1.shape[-1]
    _need(t_logits, (B, G + 1, V), U.dtype, name="t_logits", host_ok=True)
    _need(U, (B, G, V), name="U")
    _need(W1, (V, r), U.dtype, name="W1")
    _need(W2, (V, r), U.dtype, name="W2")
    _need(x0, (B,), torch.int32, name="x0")
    _need(x, (B, G), torch.int32, name="x")
    _need(lse_d, (B, G), torch.float32, name="lse_d")
    _need(logp_d, (B, G), torch.float32, name="logp_d")
    _need(ell, (B,), torch.int32, name="ell")
    dt = _dtype_code(t_logits, U, W1, W2)
    dev = W1.device
    kind = int(head["kind"])
    if kind != HEAD_MARKOV:
        _need(head["E"], (B, G, r), U.dtype, name="E")
    hs = _Head(kind, None, None, head["E"].data_ptr() if kind != HEAD_MARKOV else None)
    if out is None:
        out = dict(n_accept=torch.empty(B, dtype=torch.int32, device=dev),
                   next_token=torch.empty(B, dtype=torch.int32, device=dev))
    ws = _workspace(lib.dspark_verify_workspace_size(B, G, V, r), dev, workspace)
    _check("dspark_verify_ex",
           lib.dspark_verify_ex(B, G, V, r, dt, _ptr(t_logits), _ptr(U), _ptr(W1), _ptr(W2), _ptr(x0),
                                _ptr(x), _ptr(lse_d), _ptr(logp_d), _ptr(ell), float(temperature),
                                int(seed) & (2**64 - 1), ctypes.addressof(hs), _ptr(out["n_accept"]),
                                _ptr(out["next_token"]), _ptr(ws), _nbytes(ws), _stream(stream)))
    return out
