"""ctypes binding of ``libmoe_gb300.so`` (the C ABI in ``include/moe_gb300.h``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are ``torch`` CUDA tensors (device memory); ``None`` passes a
NULL pointer.  The stream defaults to torch's current stream.  A non-OK status
raises ``MoEError``.  There is no fallback: if the library is missing, importing
this module fails.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int32, c_int64, c_size_t, c_void_p

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_CUDA",
          -4: "MOE_ERR_WORKSPACE_TOO_SMALL", -5: "MOE_ERR_TIMEOUT", -6: "MOE_ERR_DEVICE_BOUNDS",
          -7: "MOE_ERR_MISALIGNED", -8: "MOE_ERR_RANGE", -9: "MOE_ERR_BAD_PACK"}
DTYPES = {"f32": 0, "bf16": 1}
SCORES = {"softmax": 0, "sigmoid": 1}
NORMS = {"none": 0, "l1": 1, "softmax_selected": 2, "lp": 3}
SHARED_MODES = {"none": 0, "const": 1, "gate": 2}
CAP_POLICIES = {"none": 0, "per_expert": 1, "rank_wide": 2}
H_FORMATS = {"bf16": 0, "f16": 1}


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({_lib.moe_status_string(status).decode()})")


class moe_config(ctypes.Structure):
    _fields_ = [("T", c_int64), ("d_model", c_int32), ("N", c_int32), ("K", c_int32),
                ("d_expert", c_int32), ("d_shared", c_int32), ("dtype", c_int32),
                ("score", c_int32), ("norm", c_int32), ("alpha", c_float),
                ("shared_mode", c_int32), ("shared_gain", c_float), ("cap_policy", c_int32),
                ("capacity_factor", c_double), ("num_ranks", c_int32), ("rho", POINTER(c_int32)),
                ("norm_p", c_float), ("h_format", c_int32), ("h_scale_log2", c_int32)]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("W_router", "router_bias", "selection_bias", "shared_gate_w",
                                        "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down")]


GRAD_FIELDS = ("dx", "dW_gate", "dW_up", "dW_down", "dWs_gate", "dWs_up", "dWs_down", "dW_router",
               "dshared_gate_w")


class moe_grads(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in GRAD_FIELDS]


OUTPUT_FIELDS = ("y", "topk_idx", "topk_w", "shared_coef", "logits", "counts_req", "counts_keep",
                 "offsets", "route_pos", "perm_src", "R_req", "R_keep", "drop_stats")


class moe_outputs(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in OUTPUT_FIELDS]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first "
                          "(python routing_shared_expert_gb300/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    P = c_void_p
    C = POINTER(moe_config)
    sig = {
        "moe_version": ([], c_char_p),
        "moe_status_string": ([c_int32], c_char_p),
        "moe_workspace_size": ([C, POINTER(c_size_t)], c_int32),
        "moe_workspace_init": ([P, c_size_t, P], c_int32),
        "moe_packed_weights_size": ([c_int64, POINTER(c_size_t)], c_int32),
        "moe_pack_weights": ([P, c_int64, P, c_size_t, P], c_int32),
        "moe_route": ([C, P, P, P, P, P, P, P, P, P, P, c_size_t, P], c_int32),
        "moe_balance_stats": ([C, P, P, P, P, P, P, P, P, P, c_size_t, P], c_int32),
        "moe_bias_update": ([c_int32, P, c_float, P, P], c_int32),
        "moe_permute": ([C, P, P, P, P, P, P, P, P, P, P, P, P, c_size_t, P], c_int32),
        "moe_permute_noalloc": ([C, P, P, P, P, P, P, P, P, P, P, P, P], c_int32),
        "moe_grouped_swiglu": ([C, P, P, P, P, P, P, P, P, c_size_t, P], c_int32),
        "moe_shared_mlp": ([C, P, P, P, P, P, P, c_size_t, P], c_int32),
        "moe_combine": ([C, P, P, P, P, P, P, P], c_int32),
        "moe_layer_forward": ([C, POINTER(moe_weights), P, POINTER(moe_outputs), P, c_size_t, P], c_int32),
        "moe_layer_forward_profiled": ([C, POINTER(moe_weights), P, POINTER(moe_outputs), P, c_size_t, P,
                                        POINTER(c_void_p)], c_int32),
        "moe_merge_shared": ([c_int32, c_int32, c_int32, POINTER(c_int32), POINTER(c_void_p),
                              POINTER(c_void_p), POINTER(c_void_p), P, P, P, P], c_int32),
        "moe_read_status": ([P, POINTER(c_int32), P], c_int32),
        "moe_check_wait_bound": ([P, c_size_t, c_int64, P], c_int32),
        "moe_ep_keep_matrix": ([c_int32, c_int32, c_int32, POINTER(c_int32), c_int32, c_double, P, P,
                                P, P, P, P], c_int32),
        "moe_ep_place": ([c_int32, c_int32, c_int64, c_int32, c_int32, P, P, P, P, P, P, P, c_size_t, P], c_int32),
        "moe_ep_keep_matrix_host": ([c_int32, c_int32, c_int32, POINTER(c_int32), c_int32, c_double, P,
                                     P, P, P, P], c_int32),
        "moe_ep_place_host": ([c_int32, c_int32, c_int64, c_int32, c_int32, P, P, P, P], c_int32),
        "moe_ep_send_pos": ([c_int32, c_int32, c_int64, c_int32, c_int32, POINTER(c_int32), P, P, P,
                             P, P, P, P, c_size_t, P], c_int32),
        "moe_ep_recv_rows": ([c_int32, c_int32, c_int32, POINTER(c_int32), P, P, P, c_int64, P,
                              c_size_t, P], c_int32),
        "moe_rows_copy": ([P, c_int64, P, c_int64, P, c_int64, P, c_int64, c_int64, c_int32, P,
                           c_size_t, P], c_int32),
        "moe_ep_send_pos_host": ([c_int32, c_int32, c_int64, c_int32, c_int32, POINTER(c_int32), P,
                                  P, P, P, P, P], c_int32),
        "moe_ep_recv_rows_host": ([c_int32, c_int32, c_int32, POINTER(c_int32), P, P, P, c_int64],
                                  c_int32),
        "moe_rows_copy_host": ([P, c_int64, P, c_int64, P, c_int64, P, c_int64, c_int64, c_int32],
                               c_int32),
        "moe_backward_workspace_size": ([C, POINTER(c_size_t)], c_int32),
        "moe_layer_backward": ([C, POINTER(moe_weights), P, POINTER(moe_outputs), P, POINTER(moe_grads),
                                P, c_size_t, P], c_int32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def library():
    """The loaded ``ctypes.CDLL``."""
    return _lib


def version() -> str:
    return _lib.moe_version().decode()


def _enum(table, v):
    return table[v] if isinstance(v, str) else int(v)


def make_config(T, d_model, N, K, d_expert, d_shared, dtype="bf16", score="softmax", norm="l1",
                alpha=1.0, shared_mode="const", shared_gain=1.0, cap_policy="none",
                capacity_factor=1.0, num_ranks=1, rho=None, norm_p=2.0, h_format="bf16",
                h_scale_log2=0) -> moe_config:
    """Build a ``moe_config``; ``rho`` (host list) is kept alive on the returned object."""
    c = moe_config()
    c.T, c.d_model, c.N, c.K = int(T), int(d_model), int(N), int(K)
    c.d_expert, c.d_shared = int(d_expert), int(d_shared)
    c.dtype = _enum(DTYPES, dtype)
    c.score = _enum(SCORES, score)
    c.norm = _enum(NORMS, norm)
    c.alpha = float(alpha)
    c.shared_mode = _enum(SHARED_MODES, shared_mode)
    c.shared_gain = float(shared_gain)
    c.cap_policy = _enum(CAP_POLICIES, cap_policy)
    c.capacity_factor = float(capacity_factor)
    c.num_ranks = int(num_ranks)
    c.norm_p = float(norm_p)
    c.h_format = _enum(H_FORMATS, h_format)
    c.h_scale_log2 = int(h_scale_log2)
    if rho is not None:
        arr = (c_int32 * len(rho))(*[int(v) for v in rho])
        c._rho_keepalive = arr
        c.rho = ctypes.cast(arr, POINTER(c_int32))
    return c


def copy_config(cfg: moe_config, **changes) -> moe_config:
    """A copy of ``cfg`` (sharing its host ``rho`` array) with some fields changed."""
    c = moe_config()
    ctypes.memmove(ctypes.byref(c), ctypes.byref(cfg), ctypes.sizeof(moe_config))
    if hasattr(cfg, "_rho_keepalive"):
        c._rho_keepalive = cfg._rho_keepalive
    for k, v in changes.items():
        setattr(c, k, v)
    return c


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return c_void_p(t)
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return c_void_p(stream)
    return c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status)


def moe_workspace_size(cfg: moe_config) -> int:
    n = c_size_t(0)
    _check("moe_workspace_size", _lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return int(n.value)


def moe_workspace_init(workspace, stream=None):
    _check("moe_workspace_init", _lib.moe_workspace_init(_ptr(workspace), workspace.numel(), _stream(stream)))


def alloc_workspace(cfg: moe_config, device="cuda", stream=None):
    """A zero-status workspace (uint8 tensor) large enough for every entry point of ``cfg``."""
    import torch
    ws = torch.empty(max(moe_workspace_size(cfg), 256), dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws


def moe_packed_weights_size(elements: int) -> int:
    n = c_size_t(0)
    _check("moe_packed_weights_size", _lib.moe_packed_weights_size(int(elements), ctypes.byref(n)))
    return int(n.value)


def moe_pack_weights(W, packed, stream=None):
    """Pack the bf16 tensor W into ``packed`` (uint8 device tensor) for the fp16 intermediate."""
    _check("moe_pack_weights", _lib.moe_pack_weights(_ptr(W), W.numel(), _ptr(packed), packed.numel(),
                                                     _stream(stream)))


def pack_weights(W, stream=None):
    """A new packed buffer (uint8 device tensor) holding W for the fp16 intermediate."""
    import torch
    packed = torch.empty(moe_packed_weights_size(W.numel()), dtype=torch.uint8, device=W.device)
    moe_pack_weights(W, packed, stream)
    return packed


def moe_route(cfg, x, W_router, router_bias, selection_bias, shared_gate_w, topk_idx, topk_w,
              shared_coef, logits, workspace, stream=None):
    _check("moe_route", _lib.moe_route(
        ctypes.byref(cfg), _ptr(x), _ptr(W_router), _ptr(router_bias), _ptr(selection_bias),
        _ptr(shared_gate_w), _ptr(topk_idx), _ptr(topk_w), _ptr(shared_coef), _ptr(logits),
        _ptr(workspace), workspace.numel(), _stream(stream)))


STATS = ("lbl", "imax_req", "imax_keep", "imax_rank_req", "imax_rank_keep", "ih_req", "ih_keep",
         "cv_req", "never_selected", "drop_fraction")


def moe_balance_stats(cfg, logits, counts_req, counts_keep, R_req, R_keep, P, f, stats, workspace,
                      stream=None):
    """stats: float32 [len(STATS)] device tensor, indexed as STATS."""
    _check("moe_balance_stats", _lib.moe_balance_stats(
        ctypes.byref(cfg), _ptr(logits), _ptr(counts_req), _ptr(counts_keep), _ptr(R_req),
        _ptr(R_keep), _ptr(P), _ptr(f), _ptr(stats), _ptr(workspace), workspace.numel(),
        _stream(stream)))


def moe_bias_update(N, counts, gamma, bias, stream=None):
    _check("moe_bias_update", _lib.moe_bias_update(int(N), _ptr(counts), float(gamma), _ptr(bias),
                                                    _stream(stream)))


def moe_permute(cfg, x, topk_idx, counts_req, counts_keep, offsets, route_pos, perm_src, x_perm,
                R_req, R_keep, drop_stats, workspace, stream=None):
    _check("moe_permute", _lib.moe_permute(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(counts_req), _ptr(counts_keep),
        _ptr(offsets), _ptr(route_pos), _ptr(perm_src), _ptr(x_perm), _ptr(R_req), _ptr(R_keep),
        _ptr(drop_stats), _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_permute_noalloc(cfg, x, topk_idx, counts_req, counts_keep, offsets, route_pos, perm_src,
                        x_perm, R_req, R_keep, drop_stats, stream=None):
    """moe_permute for callers that cannot allocate: no workspace (see the C header)."""
    _check("moe_permute_noalloc", _lib.moe_permute_noalloc(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(counts_req), _ptr(counts_keep),
        _ptr(offsets), _ptr(route_pos), _ptr(perm_src), _ptr(x_perm), _ptr(R_req), _ptr(R_keep),
        _ptr(drop_stats), _stream(stream)))


def moe_grouped_swiglu(cfg, x_rows, offsets, perm_src, W_gate, W_up, W_down, f, workspace,
                       stream=None):
    """x_rows is x_perm when perm_src is None, else x (rows gathered through perm_src)."""
    _check("moe_grouped_swiglu", _lib.moe_grouped_swiglu(
        ctypes.byref(cfg), _ptr(x_rows), _ptr(offsets), _ptr(perm_src), _ptr(W_gate), _ptr(W_up),
        _ptr(W_down), _ptr(f), _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_shared_mlp(cfg, x, Ws_gate, Ws_up, Ws_down, g, workspace, stream=None):
    _check("moe_shared_mlp", _lib.moe_shared_mlp(
        ctypes.byref(cfg), _ptr(x), _ptr(Ws_gate), _ptr(Ws_up), _ptr(Ws_down), _ptr(g),
        _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_combine(cfg, f, route_pos, topk_w, g, shared_coef, y, stream=None):
    _check("moe_combine", _lib.moe_combine(
        ctypes.byref(cfg), _ptr(f), _ptr(route_pos), _ptr(topk_w), _ptr(g), _ptr(shared_coef),
        _ptr(y), _stream(stream)))


def make_weights(W_router, router_bias, shared_gate_w, W_gate, W_up, W_down, Ws_gate=None,
                 Ws_up=None, Ws_down=None, selection_bias=None) -> moe_weights:
    w = moe_weights()
    keep = []
    for name, t in (("W_router", W_router), ("router_bias", router_bias),
                    ("selection_bias", selection_bias),
                    ("shared_gate_w", shared_gate_w), ("W_gate", W_gate), ("W_up", W_up),
                    ("W_down", W_down), ("Ws_gate", Ws_gate), ("Ws_up", Ws_up), ("Ws_down", Ws_down)):
        p = _ptr(t)
        setattr(w, name, p.value if p is not None else None)
        keep.append(t)
    w._keepalive = keep
    return w


def make_outputs(**tensors) -> moe_outputs:
    o = moe_outputs()
    for name in OUTPUT_FIELDS:
        t = tensors.get(name)
        p = _ptr(t)
        setattr(o, name, p.value if p is not None else None)
    o._keepalive = list(tensors.values())
    return o


def moe_layer_forward(cfg, weights: moe_weights, x, outputs: moe_outputs, workspace, stream=None):
    _check("moe_layer_forward", _lib.moe_layer_forward(
        ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), ctypes.byref(outputs), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def moe_layer_forward_profiled(cfg, weights: moe_weights, x, outputs: moe_outputs, workspace, events,
                               stream=None):
    """moe_layer_forward recording 5 torch.cuda.Event objects (created with enable_timing):
    before the router and after the router, the permutation, the routed experts and the
    shared expert + combine."""
    handles = []
    for ev in events:
        if ev.cuda_event == 0:       # torch creates the event on first record
            ev.record()
        handles.append(ev.cuda_event)
    arr = (c_void_p * 5)(*handles)
    _check("moe_layer_forward_profiled", _lib.moe_layer_forward_profiled(
        ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), ctypes.byref(outputs), _ptr(workspace),
        workspace.numel(), _stream(stream), arr))


def moe_merge_shared(d_model, dtype, gate_parts, up_parts, down_parts, Ws_gate, Ws_up, Ws_down,
                     stream=None):
    n = len(gate_parts)
    widths = (c_int32 * n)(*[int(t.shape[0]) for t in gate_parts])
    gp = (c_void_p * n)(*[t.data_ptr() for t in gate_parts])
    up = (c_void_p * n)(*[t.data_ptr() for t in up_parts])
    dp = (c_void_p * n)(*[t.data_ptr() for t in down_parts])
    _check("moe_merge_shared", _lib.moe_merge_shared(
        int(d_model), _enum(DTYPES, dtype), n, widths, gp, up, dp, _ptr(Ws_gate), _ptr(Ws_up),
        _ptr(Ws_down), _stream(stream)))


def moe_read_status(workspace, stream=None) -> int:
    code = c_int32(0)
    _check("moe_read_status", _lib.moe_read_status(_ptr(workspace), ctypes.byref(code), _stream(stream)))
    return int(code.value)


def moe_check_wait_bound(workspace, limit_ns: int, stream=None):
    """Self-check of the device wait bound (see the C header): leaves MOE_ERR_TIMEOUT in the
    workspace status word once a barrier wait of limit_ns runs out."""
    _check("moe_check_wait_bound", _lib.moe_check_wait_bound(_ptr(workspace), workspace.numel(),
                                                               int(limit_ns), _stream(stream)))


def moe_backward_workspace_size(cfg: moe_config) -> int:
    n = c_size_t(0)
    _check("moe_backward_workspace_size", _lib.moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return int(n.value)


def make_grads(**tensors) -> moe_grads:
    g = moe_grads()
    for name in GRAD_FIELDS:
        p = _ptr(tensors.get(name))
        setattr(g, name, p.value if p is not None else None)
    g._keepalive = list(tensors.values())
    return g


def moe_layer_backward(cfg, weights: moe_weights, x, fwd_outputs: moe_outputs, dy, grads: moe_grads,
                       workspace, stream=None):
    _check("moe_layer_backward", _lib.moe_layer_backward(
        ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), ctypes.byref(fwd_outputs), _ptr(dy),
        ctypes.byref(grads), _ptr(workspace), workspace.numel(), _stream(stream)))

