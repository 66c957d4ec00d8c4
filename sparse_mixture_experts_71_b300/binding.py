"""Thin ctypes binding of libmoe (the C ABI declared in include/moe.h,
include/moe_pipeline.h and include/moe_backward.h).

Argument marshalling only: every step of the layer runs in libmoe's CUDA
kernels.  PyTorch supplies device memory and the current CUDA stream.  The
functions keep the C names without the ``moe_`` prefix.

The library must have been built (``python -m sparse_mixture_experts_71_b300.build``);
importing this module without it raises, it never falls back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_F32, MOE_BF16 = 0, 1
MOE_TOKEN_CHOICE, MOE_EXPERT_CHOICE = 0, 1
MOE_DROP, MOE_REROUTE = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "misaligned pointer or row length",
          3: "workspace missing, misaligned or too small", 4: "unsupported shape",
          5: "CUDA runtime error", 6: "device-side error recorded"}

EXPORTED = ("moe_workspace_size", "moe_status_string", "moe_route", "moe_dispatch",
            "moe_expert_ffn", "moe_combine", "moe_forward", "moe_get_device_error",
            "moe_launch_count", "moe_dispatch_noalloc", "moe_check_wait_timeout",
            "moe_update_balance_bias", "moe_pipeline_workspace_size", "moe_pipeline_create",
            "moe_pipeline_submit", "moe_pipeline_join", "moe_pipeline_destroy",
            "moe_route_expert_choice", "moe_expert_choice_capacity",
            "moe_backward_workspace_size", "moe_backward", "moe_check_segment_maps")


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("renormalize", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("routing", ctypes.c_int32),
                ("overflow", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {STATUS.get(status, 'unknown status')} (status {status})")
        self.status = status


_P = ctypes.c_void_p
_lib = None


def load() -> ctypes.CDLL:
    """Load libmoe.so once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"libmoe.so is not built ({_LIB_PATH}); run "
                              "python -m sparse_mixture_experts_71_b300.build")
        lib = ctypes.CDLL(_LIB_PATH)
        lib.moe_workspace_size.restype = ctypes.c_size_t
        lib.moe_workspace_size.argtypes = [ctypes.POINTER(MoeConfig)]
        lib.moe_status_string.restype = ctypes.c_char_p
        lib.moe_status_string.argtypes = [ctypes.c_int]
        cfgp = ctypes.POINTER(MoeConfig)
        sz = ctypes.c_size_t
        lib.moe_route.argtypes = [cfgp] + [_P] * 11 + [_P, sz, _P]
        lib.moe_dispatch.argtypes = [cfgp] + [_P] * 8 + [_P, sz, _P]
        lib.moe_expert_ffn.argtypes = [cfgp] + [_P] * 8 + [_P, sz, _P]
        lib.moe_combine.argtypes = [cfgp, _P, _P, _P, _P]
        lib.moe_forward.argtypes = [cfgp] + [_P] * 13 + [_P, sz, _P]
        lib.moe_get_device_error.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_int32),
                                             ctypes.POINTER(ctypes.c_int32)]
        for name in EXPORTED[2:8]:
            getattr(lib, name).restype = ctypes.c_int
        lib.moe_dispatch_noalloc.restype = ctypes.c_int
        lib.moe_dispatch_noalloc.argtypes = [cfgp] + [_P] * 8 + [_P]
        lib.moe_launch_count.restype = ctypes.c_uint64
        lib.moe_launch_count.argtypes = []
        lib.moe_check_wait_timeout.restype = ctypes.c_int
        lib.moe_check_wait_timeout.argtypes = [_P, ctypes.c_uint64, _P]
        lib.moe_update_balance_bias.restype = ctypes.c_int
        lib.moe_update_balance_bias.argtypes = [cfgp, _P, _P, ctypes.c_float, _P]
        lib.moe_route_expert_choice.restype = ctypes.c_int
        lib.moe_route_expert_choice.argtypes = [cfgp] + [_P] * 13 + [_P, sz, _P]
        lib.moe_expert_choice_capacity.restype = ctypes.c_int32
        lib.moe_expert_choice_capacity.argtypes = [cfgp]
        lib.moe_backward_workspace_size.restype = ctypes.c_size_t
        lib.moe_backward_workspace_size.argtypes = [cfgp]
        lib.moe_check_segment_maps.restype = ctypes.c_int
        lib.moe_check_segment_maps.argtypes = [_P, sz, _P]
        lib.moe_backward.restype = ctypes.c_int
        lib.moe_backward.argtypes = ([cfgp] + [_P] * 8 + [ctypes.c_float, ctypes.c_float]
                                     + [_P] * 7 + [sz, _P])
        lib.moe_pipeline_workspace_size.restype = ctypes.c_size_t
        lib.moe_pipeline_workspace_size.argtypes = [cfgp, ctypes.c_int32]
        lib.moe_pipeline_create.restype = ctypes.c_int
        lib.moe_pipeline_create.argtypes = [cfgp, ctypes.c_int32] + [_P] * 7 + [sz, _P,
                                                                               ctypes.POINTER(_P)]
        lib.moe_pipeline_submit.restype = ctypes.c_int
        lib.moe_pipeline_submit.argtypes = [_P, _P, _P, _P]
        lib.moe_pipeline_join.restype = ctypes.c_int
        lib.moe_pipeline_join.argtypes = [_P]
        lib.moe_pipeline_destroy.restype = ctypes.c_int
        lib.moe_pipeline_destroy.argtypes = [_P]
        _lib = lib
    return _lib


def config(T, d, d_ff, E, k, dtype="bf16", capacity=None, renormalize=True,
           n_shared=0, routing="token", overflow="drop") -> MoeConfig:
    """routing: "token" (each token picks its top-k experts) or "expert" (each
    expert picks its top-C tokens); overflow: "drop" or "reroute" (a slot the
    cap drops is offered to the token's next-best expert)."""
    if routing not in ("token", "expert"):
        raise ValueError(f"routing must be 'token' or 'expert', not {routing!r}")
    if overflow not in ("drop", "reroute"):
        raise ValueError(f"overflow must be 'drop' or 'reroute', not {overflow!r}")
    return MoeConfig(T, d, d_ff, E, k, MOE_BF16 if dtype == "bf16" else MOE_F32,
                     -1 if capacity is None else int(capacity), 1 if renormalize else 0,
                     int(n_shared), MOE_EXPERT_CHOICE if routing == "expert" else MOE_TOKEN_CHOICE,
                     MOE_REROUTE if overflow == "reroute" else MOE_DROP)


def ranked_columns(cfg: MoeConfig) -> int:
    """Columns of moe_route's topk_idx / topk_w: k, or min(2k, E) when
    rerouting (the k choices, then the next-best experts)."""
    return min(2 * cfg.k, cfg.E) if cfg.overflow == MOE_REROUTE else cfg.k + cfg.n_shared


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(fn, st):
    if st != 0:
        raise MoeError(fn, st)


def workspace_size(cfg: MoeConfig) -> int:
    return int(load().moe_workspace_size(ctypes.byref(cfg)))


def workspace(cfg: MoeConfig, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (the device error record must start at zero)."""
    n = workspace_size(cfg)
    if n == 0:
        raise MoeError("moe_workspace_size", 1)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def route(cfg, x, W_r, topk_idx, topk_w, ws, logit_bias=None, logits_in=None, logits_out=None,
          expert_counts=None, aux_out=None, z_loss_out=None, logit_noise=None, stream=None):
    _check("moe_route", load().moe_route(
        ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(logit_bias), _ptr(logit_noise),
        _ptr(logits_in), _ptr(logits_out),
        _ptr(topk_idx), _ptr(topk_w), _ptr(expert_counts), _ptr(aux_out), _ptr(z_loss_out),
        _ptr(ws), ws.numel(), _stream(stream)))


def dispatch(cfg, x, topk_idx, offsets, slot_of, perm_token, x_perm, ws, topk_w=None,
             perm_w=None, stream=None):
    _check("moe_dispatch", load().moe_dispatch(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(offsets), _ptr(slot_of),
        _ptr(perm_token), _ptr(perm_w), _ptr(x_perm), _ptr(ws), ws.numel(), _stream(stream)))


def expert_ffn(cfg, x_perm, offsets, W1, b1, W2, b2, y_perm, ws, perm_w=None, stream=None):
    _check("moe_expert_ffn", load().moe_expert_ffn(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2),
        _ptr(perm_w), _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)))


def dispatch_noalloc(cfg, x, topk_idx, offsets, slot_of, perm_token, x_perm, topk_w=None,
                     perm_w=None, stream=None):
    """moe_dispatch_noalloc: dispatch with the library's own fixed scratch array
    (no workspace argument; T * k <= 65536, E <= 256)."""
    _check("moe_dispatch_noalloc", load().moe_dispatch_noalloc(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(offsets), _ptr(slot_of),
        _ptr(perm_token), _ptr(perm_w), _ptr(x_perm), _stream(stream)))


def combine(cfg, y_perm, slot_of, y, stream=None):
    _check("moe_combine", load().moe_combine(
        ctypes.byref(cfg), _ptr(y_perm), _ptr(slot_of), _ptr(y), _stream(stream)))


def forward(cfg, x, W_r, W1, b1, W2, b2, y, ws, logit_bias=None, aux_out=None,
            expert_counts=None, logits_out=None, z_loss_out=None, logit_noise=None,
            stream=None):
    _check("moe_forward", load().moe_forward(
        ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(logit_bias), _ptr(logit_noise), _ptr(W1),
        _ptr(b1), _ptr(W2),
        _ptr(b2), _ptr(y), _ptr(aux_out), _ptr(expert_counts), _ptr(logits_out),
        _ptr(z_loss_out), _ptr(ws), ws.numel(), _stream(stream)))


def route_expert_choice(cfg, x, W_r, offsets, perm_token, perm_w, slot_of, ws, x_perm=None,
                        logit_bias=None, logit_noise=None, logits_in=None, logits_out=None,
                        expert_counts=None, z_loss_out=None, stream=None):
    """Expert-choice route + dispatch: every expert's top-C tokens, the rows
    (offsets [E+1], perm_token / perm_w [E*C], slot_of [T][E]) and, with
    x_perm [E*C][d], the gathered rows."""
    _check("moe_route_expert_choice", load().moe_route_expert_choice(
        ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(logit_bias), _ptr(logit_noise),
        _ptr(logits_in), _ptr(logits_out), _ptr(offsets), _ptr(perm_token), _ptr(perm_w),
        _ptr(slot_of), _ptr(x_perm), _ptr(expert_counts), _ptr(z_loss_out), _ptr(ws),
        ws.numel(), _stream(stream)))


def expert_choice_capacity(cfg: MoeConfig) -> int:
    """C, the tokens each expert takes under expert-choice routing."""
    return int(load().moe_expert_choice_capacity(ctypes.byref(cfg)))


def backward_workspace(cfg: MoeConfig, device="cuda") -> torch.Tensor:
    """A zero-filled workspace for moe_backward."""
    n = int(load().moe_backward_workspace_size(ctypes.byref(cfg)))
    if n == 0:
        raise MoeError("moe_backward_workspace_size", 4)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def backward(cfg, x, W_r, W1, b1, W2, b2, dy, dx, dW_r, dW1, db1, dW2, db2, ws, logit_bias=None,
             aux_grad: float = 0.0, z_grad: float = 0.0, stream=None):
    """Gradients of <dy, y> + aux_grad aux + z_grad z_loss (moe_backward):
    dx (layer dtype), dW_r, dW1, db1, dW2, db2 (fp32), written in place."""
    _check("moe_backward", load().moe_backward(
        ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(logit_bias), _ptr(W1), _ptr(b1), _ptr(W2),
        _ptr(b2), _ptr(dy), ctypes.c_float(aux_grad), ctypes.c_float(z_grad), _ptr(dx),
        _ptr(dW_r), _ptr(dW1), _ptr(db1), _ptr(dW2), _ptr(db2), _ptr(ws), ws.numel(),
        _stream(stream)))


def launch_count() -> int:
    """Kernels libmoe has enqueued in this process (diagnostics)."""
    return int(load().moe_launch_count())


def update_balance_bias(cfg, expert_counts, logit_bias, step: float, stream=None) -> None:
    """Auxiliary-loss-free balancing step on logit_bias (in place) from the
    per-expert assignment counts of a routed batch."""
    _check("moe_update_balance_bias", load().moe_update_balance_bias(
        ctypes.byref(cfg), _ptr(expert_counts), _ptr(logit_bias), ctypes.c_float(step),
        _stream(stream)))


def check_wait_timeout(ws, timeout_ns: int, stream=None) -> None:
    """Run one bounded pipeline wait that times out (diagnostics); the time-out
    is recorded in ws's error record (read it with get_device_error)."""
    _check("moe_check_wait_timeout",
           load().moe_check_wait_timeout(_ptr(ws), ctypes.c_uint64(timeout_ns), _stream(stream)))


def check_segment_maps(ws, stream=None) -> None:
    """Check the device-side edits of the per-segment tensor maps the backward
    pass's weight-gradient products use against the driver's encoding
    (diagnostics; ws: a device buffer of at least 3 MiB; synchronises)."""
    _check("moe_check_segment_maps", load().moe_check_segment_maps(
        _ptr(ws), ctypes.c_size_t(ws.numel() * ws.element_size()), _stream(stream)))


def get_device_error(ws, stream=None):
    """(status, code, info): synchronises the stream, reads and clears the record."""
    code, info = ctypes.c_int32(0), ctypes.c_int32(0)
    st = load().moe_get_device_error(_ptr(ws), _stream(stream), ctypes.byref(code),
                                     ctypes.byref(info))
    return st, code.value, info.value


def pipeline_workspace_size(cfg: MoeConfig, depth: int = 2) -> int:
    return int(load().moe_pipeline_workspace_size(ctypes.byref(cfg), depth))


class Pipeline:
    """Host-buffer executor (moe_pipeline_*): batches of cfg.T tokens in host
    memory in, y and the auxiliary loss to host memory out, the copies of
    neighbouring batches overlapping the forward pass on ``stream``.

    Keeps the workspace it allocates (and the weights it is given) alive;
    ``close()`` (or garbage collection) destroys the executor."""

    def __init__(self, cfg: MoeConfig, W_r, W1, b1, W2, b2, logit_bias=None, depth: int = 2,
                 stream=None, device="cuda"):
        n = pipeline_workspace_size(cfg, depth)
        if n == 0:
            raise MoeError("moe_pipeline_workspace_size", 1)
        self.cfg, self.depth = cfg, depth
        self.ws = torch.zeros(n, dtype=torch.uint8, device=device)
        self._keep = (W_r, W1, b1, W2, b2, logit_bias)
        self._stream = stream
        h = _P()
        _check("moe_pipeline_create", load().moe_pipeline_create(
            ctypes.byref(cfg), depth, _ptr(W_r), _ptr(logit_bias), _ptr(W1), _ptr(b1), _ptr(W2),
            _ptr(b2), _ptr(self.ws), n, _stream(stream), ctypes.byref(h)))
        self._h = h

    def submit(self, x_host, y_host, aux_host=None) -> None:
        """Enqueue one batch; x_host / y_host (T, d) and aux_host (1,) are host
        tensors (pinned for overlap) that must stay alive until after join()."""
        _check("moe_pipeline_submit", load().moe_pipeline_submit(
            self._h, _ptr(x_host), _ptr(y_host), _ptr(aux_host)))

    def join(self) -> None:
        """The stream waits for the outputs of every submitted batch."""
        _check("moe_pipeline_join", load().moe_pipeline_join(self._h))

    def close(self) -> None:
        if getattr(self, "_h", None):
            st = load().moe_pipeline_destroy(self._h)
            self._h = None
            _check("moe_pipeline_destroy", st)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
