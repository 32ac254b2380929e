"""Thin ctypes binding of libspec_verify.so (declared in include/spec_verify.h).

Argument marshalling only: shapes, dtypes and devices are checked, outputs and
a per-stream workspace are allocated with torch, and raw device pointers go to
the C ABI.  Every step of the verification runs in the library's CUDA
kernels.  There is no CPU fallback: if the library cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import NamedTuple, Optional

import torch

from . import _build

(SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_CUDA, SV_ERR_DEVICE_INPUT, SV_ERR_TIMEOUT,
 SV_ERR_SCRATCH_LIMIT) = range(7)
SV_STATIC_SCRATCH_BYTES = 4 << 20
SV_F32, SV_BF16 = 0, 1

# Every function declared in include/spec_verify.h.
EXPORTED = (
    "spec_verify_abi_version", "spec_verify_workspace_size", "spec_verify_workspace_init",
    "spec_verify_dense", "spec_verify_sparse", "spec_verify_anyorder", "spec_verify_check",
    "spec_verify_status_string", "spec_verify_dense_static", "spec_verify_greedy",
    "spec_commit_confident", "spec_support_topk", "spec_verify_anyorder_rounds",
    "spec_anyorder_window",
)


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Load libspec_verify.so (raises if it is missing and not built here)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
            _build.build()
        lib = ctypes.CDLL(path)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.spec_verify_abi_version.restype = I
        lib.spec_verify_abi_version.argtypes = []
        lib.spec_verify_workspace_size.restype = Z
        lib.spec_verify_workspace_size.argtypes = [I, I, I]
        lib.spec_verify_workspace_init.restype = I
        lib.spec_verify_workspace_init.argtypes = [P, Z, P]
        lib.spec_verify_dense.restype = I
        lib.spec_verify_dense.argtypes = [P, P, I, P, P, P, I, I, I, P, P, P, P, P, Z, P]
        lib.spec_verify_sparse.restype = I
        lib.spec_verify_sparse.argtypes = [P, P, I, P, P, I, P, P, P, I, I, I, P, P, P, P, P, Z, P]
        lib.spec_verify_anyorder.restype = I
        lib.spec_verify_anyorder.argtypes = [P, P, I, P, P, P, P, I, I, I, I, P, P, P, P, P, Z, P]
        lib.spec_verify_check.restype = I
        lib.spec_verify_check.argtypes = [P, Z, P]
        lib.spec_verify_status_string.restype = ctypes.c_char_p
        lib.spec_verify_status_string.argtypes = [I]
        lib.spec_verify_greedy.restype = I
        lib.spec_verify_greedy.argtypes = [P, I, P, I, I, I, P, P, P, Z, P]
        lib.spec_commit_confident.restype = I
        lib.spec_commit_confident.argtypes = [P, I, P, ctypes.c_float, I, I, I, P, P, P, P, Z, P]
        lib.spec_support_topk.restype = I
        lib.spec_support_topk.argtypes = [P, I, I, I, ctypes.c_float, I, ctypes.c_float, P, P, P, Z, P]
        lib.spec_verify_anyorder_rounds.restype = I
        lib.spec_verify_anyorder_rounds.argtypes = [P, P, I, P, P, P, P, P, P, I, I, I, I, P, P, P, P, Z, P]
        lib.spec_anyorder_window.restype = I
        lib.spec_anyorder_window.argtypes = [I, I, ctypes.c_float]
        lib.spec_verify_dense_static.restype = I
        lib.spec_verify_dense_static.argtypes = [P, P, I, P, P, P, I, I, I, P, P, P, P, P]
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().spec_verify_status_string(int(status)).decode()


def abi_version() -> int:
    return int(load().spec_verify_abi_version())


def workspace_size(B: int, gamma_or_W: int, V: int) -> int:
    return int(load().spec_verify_workspace_size(int(B), int(gamma_or_W), int(V)))


# ---------------------------------------------------------------------------
# workspace cache: one zero-initialised buffer per (device, stream)
# ---------------------------------------------------------------------------
_ws_cache: dict = {}


def _stream_ptr(stream: Optional[torch.cuda.Stream], device: torch.device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def get_workspace(nbytes: int, device: torch.device, stream_ptr: int) -> torch.Tensor:
    """A zeroed workspace of at least nbytes for calls on this stream.  The
    library leaves it zeroed after every successful call, so it is reused."""
    key = (device.index, stream_ptr)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        rc = load().spec_verify_workspace_init(ws.data_ptr(), ws.numel(), stream_ptr)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_workspace_init")
        _ws_cache[key] = ws
    return ws


def check(device=None, stream: Optional[torch.cuda.Stream] = None) -> int:
    """spec_verify_check on the cached workspace of this stream (syncs)."""
    if device is None:
        device = torch.device("cuda", torch.cuda.current_device())
    elif not isinstance(device, torch.device):
        device = torch.device("cuda", int(device))
    sp = _stream_ptr(stream, device)
    ws = _ws_cache.get((device.index, sp))
    if ws is None:
        return SV_OK
    return int(load().spec_verify_check(ws.data_ptr(), ws.numel(), sp))


class VerifyResult(NamedTuple):
    n_accepted: torch.Tensor
    out_tokens: torch.Tensor
    residual: Optional[torch.Tensor]
    accept_prob: Optional[torch.Tensor]


def _req(t: torch.Tensor, name: str, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _logit_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def spec_verify_dense(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                      draft_ids: torch.Tensor, u_accept: torch.Tensor, u_sample: torch.Tensor,
                      *, residual: bool = False, accept_prob: bool = False,
                      out: Optional[VerifyResult] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> VerifyResult:
    """Dense verification.  target [B, g+1, V], draft [B, g, V] (bf16 or fp32,
    CUDA), draft_ids [B, g] int32, u_accept [B, g] fp32, u_sample [B] fp32."""
    lib = load()
    dev = target_logits.device
    if dev.type != "cuda":
        raise ValueError("spec_verify_dense needs CUDA tensors")
    dt = _logit_dtype(target_logits)
    B, G1, V = target_logits.shape
    G = G1 - 1
    _req(target_logits, "target_logits", target_logits.dtype, (B, G + 1, V), dev)
    _req(draft_logits, "draft_logits", target_logits.dtype, (B, G, V), dev)
    _req(draft_ids, "draft_ids", torch.int32, (B, G), dev)
    _req(u_accept, "u_accept", torch.float32, (B, G), dev)
    _req(u_sample, "u_sample", torch.float32, (B,), dev)
    if out is None:
        out = VerifyResult(
            torch.empty(B, dtype=torch.int32, device=dev),
            torch.empty(B, G + 1, dtype=torch.int32, device=dev),
            torch.empty(B, V, dtype=torch.float32, device=dev) if residual else None,
            torch.empty(B, G, dtype=torch.float32, device=dev) if accept_prob else None)
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(workspace_size(B, G, V), dev, sp)
    with torch.cuda.device(dev):
        rc = lib.spec_verify_dense(
            _ptr(target_logits), _ptr(draft_logits) if G > 0 else None, dt, _ptr(draft_ids),
            _ptr(u_accept), _ptr(u_sample), B, G, V, _ptr(out.n_accepted), _ptr(out.out_tokens),
            _ptr(out.residual), _ptr(out.accept_prob), ws.data_ptr(), ws.numel(), sp)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_dense")
    return out


def spec_verify_greedy(target_logits: torch.Tensor, draft_ids: torch.Tensor, *,
                       out: Optional[VerifyResult] = None,
                       stream: Optional[torch.cuda.Stream] = None) -> VerifyResult:
    """Greedy (T = 0) verification.  target [B, g+1, V] (bf16 or fp32, CUDA),
    draft_ids [B, g] int32.  Returns n_accepted and out_tokens."""
    lib = load()
    dev = target_logits.device
    if dev.type != "cuda":
        raise ValueError("spec_verify_greedy needs CUDA tensors")
    dt = _logit_dtype(target_logits)
    B, G1, V = target_logits.shape
    G = G1 - 1
    _req(target_logits, "target_logits", target_logits.dtype, (B, G + 1, V), dev)
    _req(draft_ids, "draft_ids", torch.int32, (B, G), dev)
    if out is None:
        out = VerifyResult(torch.empty(B, dtype=torch.int32, device=dev),
                           torch.empty(B, G + 1, dtype=torch.int32, device=dev), None, None)
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(workspace_size(B, G, V), dev, sp)
    with torch.cuda.device(dev):
        rc = lib.spec_verify_greedy(_ptr(target_logits), dt, _ptr(draft_ids) if G > 0 else None,
                                    B, G, V, _ptr(out.n_accepted), _ptr(out.out_tokens),
                                    ws.data_ptr(), ws.numel(), sp)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_greedy")
    return out


class CommitResult(NamedTuple):
    commit: torch.Tensor
    tokens: torch.Tensor
    confidence: Optional[torch.Tensor]


def spec_commit_confident(logits: torch.Tensor, masked: torch.Tensor, tau: float, *,
                          confidence: bool = False, out: Optional[CommitResult] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> CommitResult:
    """Confidence-threshold commit of B blocks.  logits [B, W, V] (bf16 or fp32,
    CUDA), masked [B, W] int32 (nonzero: still masked), threshold tau."""
    lib = load()
    dev = logits.device
    if dev.type != "cuda":
        raise ValueError("spec_commit_confident needs CUDA tensors")
    dt = _logit_dtype(logits)
    B, W, V = logits.shape
    _req(logits, "logits", logits.dtype, (B, W, V), dev)
    _req(masked, "masked", torch.int32, (B, W), dev)
    if out is None:
        out = CommitResult(torch.empty(B, W, dtype=torch.int32, device=dev),
                           torch.empty(B, W, dtype=torch.int32, device=dev),
                           torch.empty(B, W, dtype=torch.float32, device=dev) if confidence else None)
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(workspace_size(B, W - 1, V), dev, sp)
    with torch.cuda.device(dev):
        rc = lib.spec_commit_confident(_ptr(logits), dt, _ptr(masked), float(tau), B, W, V,
                                       _ptr(out.commit), _ptr(out.tokens), _ptr(out.confidence),
                                       ws.data_ptr(), ws.numel(), sp)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_commit_confident")
    return out


def prepare_commit(logits, masked, tau: float, out: CommitResult,
                   stream: Optional[torch.cuda.Stream] = None) -> PreparedCall:
    """Validate once and return a PreparedCall repeating spec_commit_confident."""
    spec_commit_confident(logits, masked, tau, out=out, stream=stream)
    lib = load()
    dev = logits.device
    B, W, V = logits.shape
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(workspace_size(B, W - 1, V), dev, sp)
    args = (_ptr(logits), _logit_dtype(logits), _ptr(masked), ctypes.c_float(float(tau)), B, W, V,
            _ptr(out.commit), _ptr(out.tokens), _ptr(out.confidence), ws.data_ptr(), ws.numel(), sp)
    keep = (logits, masked, out, ws)
    return PreparedCall(lib.spec_commit_confident, args, keep, "spec_commit_confident")


class SupportResult(NamedTuple):
    ids: torch.Tensor
    probs: torch.Tensor


def spec_support_topk(logits: torch.Tensor, temperature: float, top_k: int, top_p: float, *,
                      out: Optional[SupportResult] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> SupportResult:
    """Sparse support lists from dense logits [..., V] (bf16 or fp32, CUDA):
    ids [..., top_k] ascending, probs [..., top_k]."""
    lib = load()
    dev = logits.device
    if dev.type != "cuda":
        raise ValueError("spec_support_topk needs CUDA tensors")
    dt = _logit_dtype(logits)
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    lead = tuple(logits.shape[:-1])
    V = int(logits.shape[-1])
    N = 1
    for d in lead:
        N *= int(d)
    K = int(top_k)
    if out is None:
        out = SupportResult(torch.empty(lead + (K,), dtype=torch.int32, device=dev),
                            torch.empty(lead + (K,), dtype=torch.float32, device=dev))
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(256, dev, sp)
    with torch.cuda.device(dev):
        rc = lib.spec_support_topk(_ptr(logits), dt, N, V, float(temperature), K, float(top_p),
                                   _ptr(out.ids), _ptr(out.probs), ws.data_ptr(), ws.numel(), sp)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_support_topk")
    return out


def prepare_support(logits, temperature: float, top_k: int, top_p: float, out: SupportResult,
                    stream: Optional[torch.cuda.Stream] = None) -> PreparedCall:
    """Validate once and return a PreparedCall repeating spec_support_topk."""
    spec_support_topk(logits, temperature, top_k, top_p, out=out, stream=stream)
    lib = load()
    dev = logits.device
    V = int(logits.shape[-1])
    N = logits.numel() // V
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(256, dev, sp)
    args = (_ptr(logits), _logit_dtype(logits), N, V, ctypes.c_float(float(temperature)),
            int(top_k), ctypes.c_float(float(top_p)), _ptr(out.ids), _ptr(out.probs),
            ws.data_ptr(), ws.numel(), sp)
    keep = (logits, out, ws)
    return PreparedCall(lib.spec_support_topk, args, keep, "spec_support_topk")


def prepare_greedy(target_logits, draft_ids, out: VerifyResult,
                   stream: Optional[torch.cuda.Stream] = None) -> PreparedCall:
    """Validate once (by running the checked call) and return a PreparedCall
    that repeats spec_verify_greedy on the same buffers."""
    spec_verify_greedy(target_logits, draft_ids, out=out, stream=stream)
    lib = load()
    dev = target_logits.device
    B, G1, V = target_logits.shape
    G = G1 - 1
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(workspace_size(B, G, V), dev, sp)
    args = (_ptr(target_logits), _logit_dtype(target_logits), _ptr(draft_ids) if G > 0 else None,
            B, G, V, _ptr(out.n_accepted), _ptr(out.out_tokens), ws.data_ptr(), ws.numel(), sp)
    keep = (target_logits, draft_ids, out, ws)
    return PreparedCall(lib.spec_verify_greedy, args, keep, "spec_verify_greedy")


def spec_verify_dense_static(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                             draft_ids: torch.Tensor, u_accept: torch.Tensor,
                             u_sample: torch.Tensor, out: VerifyResult,
                             stream: Optional[torch.cuda.Stream] = None) -> VerifyResult:
    """spec_verify_dense on the library's static scratch, for callers that
    cannot allocate: the outputs are the caller's (``out``), nothing is
    allocated here or in the library."""
    lib = load()
    dev = target_logits.device
    if dev.type != "cuda":
        raise ValueError("spec_verify_dense_static needs CUDA tensors")
    dt = _logit_dtype(target_logits)
    B, G1, V = target_logits.shape
    G = G1 - 1
    _req(target_logits, "target_logits", target_logits.dtype, (B, G + 1, V), dev)
    _req(draft_logits, "draft_logits", target_logits.dtype, (B, G, V), dev)
    _req(draft_ids, "draft_ids", torch.int32, (B, G), dev)
    _req(u_accept, "u_accept", torch.float32, (B, G), dev)
    _req(u_sample, "u_sample", torch.float32, (B,), dev)
    _req(out.n_accepted, "n_accepted", torch.int32, (B,), dev)
    _req(out.out_tokens, "out_tokens", torch.int32, (B, G + 1), dev)
    if out.residual is not None:
        _req(out.residual, "residual", torch.float32, (B, V), dev)
    if out.accept_prob is not None:
        _req(out.accept_prob, "accept_prob", torch.float32, (B, G), dev)
    sp = _stream_ptr(stream, dev)
    with torch.cuda.device(dev):
        rc = lib.spec_verify_dense_static(
            _ptr(target_logits), _ptr(draft_logits) if G > 0 else None, dt, _ptr(draft_ids),
            _ptr(u_accept), _ptr(u_sample), B, G, V, _ptr(out.n_accepted), _ptr(out.out_tokens),
            _ptr(out.residual), _ptr(out.accept_prob), sp)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_dense_static")
    return out


def spec_verify_sparse(tgt_ids: torch.Tensor, tgt_probs: torch.Tensor, drf_ids: torch.Tensor,
                       drf_probs: torch.Tensor, draft_tokens: torch.Tensor, u_accept: torch.Tensor,
                       u_sample: torch.Tensor, vocab_size: int, *, residual: bool = False,
                       accept_prob: bool = False, out: Optional[VerifyResult] = None,
                       stream: Optional[torch.cuda.Stream] = None) -> VerifyResult:
    """Sparse top-k verification.  tgt_* [B, g+1, kt], drf_* [B, g, kd]; ids
    int32 sorted ascending, probs fp32."""
    lib = load()
    dev = tgt_ids.device
    if dev.type != "cuda":
        raise ValueError("spec_verify_sparse needs CUDA tensors")
    B, G1, kt = tgt_ids.shape
    G = G1 - 1
    kd = drf_ids.shape[2] if drf_ids.dim() == 3 else 1
    _req(tgt_ids, "tgt_ids", torch.int32, (B, G + 1, kt), dev)
    _req(tgt_probs, "tgt_probs", torch.float32, (B, G + 1, kt), dev)
    _req(drf_ids, "drf_ids", torch.int32, (B, G, kd), dev)
    _req(drf_probs, "drf_probs", torch.float32, (B, G, kd), dev)
    _req(draft_tokens, "draft_tokens", torch.int32, (B, G), dev)
    _req(u_accept, "u_accept", torch.float32, (B, G), dev)
    _req(u_sample, "u_sample", torch.float32, (B,), dev)
    if out is None:
        out = VerifyResult(
            torch.empty(B, dtype=torch.int32, device=dev),
            torch.empty(B, G + 1, dtype=torch.int32, device=dev),
            torch.empty(B, kt, dtype=torch.float32, device=dev) if residual else None,
            torch.empty(B, G, dtype=torch.float32, device=dev) if accept_prob else None)
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(256, dev, sp)
    with torch.cuda.device(dev):
        rc = lib.spec_verify_sparse(
            _ptr(tgt_ids), _ptr(tgt_probs), kt, _ptr(drf_ids) if G else None,
            _ptr(drf_probs) if G else None, kd, _ptr(draft_tokens) if G else None,
            _ptr(u_accept) if G else None, _ptr(u_sample), B, G, int(vocab_size),
            _ptr(out.n_accepted), _ptr(out.out_tokens), _ptr(out.residual), _ptr(out.accept_prob),
            ws.data_ptr(), ws.numel(), sp)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_sparse")
    return out


def spec_verify_anyorder(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                         order: torch.Tensor, draft_tokens: torch.Tensor, u_accept: torch.Tensor,
                         u_sample: torch.Tensor, *, out_tokens: Optional[torch.Tensor] = None,
                         residual: bool = False, accept_prob: bool = False,
                         stream: Optional[torch.cuda.Stream] = None) -> VerifyResult:
    """Any-order verification.  target/draft [B, D, V], order [B, W] int32,
    draft_tokens [B, D] int32, u_accept [B, W], u_sample [B].  out_tokens
    [B, D] is updated in place at the window positions (allocated filled with
    -1 if not given)."""
    lib = load()
    dev = target_logits.device
    if dev.type != "cuda":
        raise ValueError("spec_verify_anyorder needs CUDA tensors")
    dt = _logit_dtype(target_logits)
    B, D, V = target_logits.shape
    W = order.shape[1]
    _req(target_logits, "target_logits", target_logits.dtype, (B, D, V), dev)
    _req(draft_logits, "draft_logits", target_logits.dtype, (B, D, V), dev)
    _req(order, "order", torch.int32, (B, W), dev)
    _req(draft_tokens, "draft_tokens", torch.int32, (B, D), dev)
    _req(u_accept, "u_accept", torch.float32, (B, W), dev)
    _req(u_sample, "u_sample", torch.float32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.full((B, D), -1, dtype=torch.int32, device=dev)
    _req(out_tokens, "out_tokens", torch.int32, (B, D), dev)
    res = VerifyResult(
        torch.empty(B, dtype=torch.int32, device=dev), out_tokens,
        torch.empty(B, V, dtype=torch.float32, device=dev) if residual else None,
        torch.empty(B, W, dtype=torch.float32, device=dev) if accept_prob else None)
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(256, dev, sp)
    with torch.cuda.device(dev):
        rc = lib.spec_verify_anyorder(
            _ptr(target_logits), _ptr(draft_logits), dt, _ptr(order), _ptr(draft_tokens),
            _ptr(u_accept), _ptr(u_sample), B, D, W, V, _ptr(res.n_accepted), _ptr(out_tokens),
            _ptr(res.residual), _ptr(res.accept_prob), ws.data_ptr(), ws.numel(), sp)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_anyorder")
    return res


class RoundsResult(NamedTuple):
    tokens: torch.Tensor         # [B, D] int32, revealed tokens written at their positions
    n_revealed: torch.Tensor     # [B] int32
    round_accepts: torch.Tensor  # [B, R] int32


def _rounds_args(target_logits, draft_logits, order, revealed, window, draft_tokens, u_accept,
                 u_sample, out: RoundsResult, ws, sp):
    B, R, D, V = (int(v) for v in target_logits.shape)
    return (_ptr(target_logits), _ptr(draft_logits), _logit_dtype(target_logits), _ptr(order),
            _ptr(revealed), _ptr(window), _ptr(draft_tokens), _ptr(u_accept), _ptr(u_sample),
            B, R, D, V, _ptr(out.tokens), _ptr(out.n_revealed), _ptr(out.round_accepts),
            ws.data_ptr(), ws.numel(), sp)


def spec_verify_anyorder_rounds(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                                order: torch.Tensor, revealed: torch.Tensor, window: torch.Tensor,
                                draft_tokens: torch.Tensor, u_accept: torch.Tensor,
                                u_sample: torch.Tensor, *, tokens: Optional[torch.Tensor] = None,
                                out: Optional[RoundsResult] = None,
                                stream: Optional[torch.cuda.Stream] = None) -> RoundsResult:
    """Windowed multi-round any-order verification.  target [B, R, D, V],
    draft [B, D, V], order [B, D], revealed [B], window [B], draft_tokens
    [B, R, D], u_accept [B, R, D] (by sigma index), u_sample [B, R].  tokens
    [B, D] is updated in place at the revealed positions (allocated filled
    with -1 if not given)."""
    lib = load()
    dev = target_logits.device
    if dev.type != "cuda":
        raise ValueError("spec_verify_anyorder_rounds needs CUDA tensors")
    B, R, D, V = target_logits.shape
    _req(target_logits, "target_logits", target_logits.dtype, (B, R, D, V), dev)
    _logit_dtype(target_logits)
    _req(draft_logits, "draft_logits", target_logits.dtype, (B, D, V), dev)
    _req(order, "order", torch.int32, (B, D), dev)
    _req(revealed, "revealed", torch.int32, (B,), dev)
    _req(window, "window", torch.int32, (B,), dev)
    _req(draft_tokens, "draft_tokens", torch.int32, (B, R, D), dev)
    _req(u_accept, "u_accept", torch.float32, (B, R, D), dev)
    _req(u_sample, "u_sample", torch.float32, (B, R), dev)
    if out is None:
        if tokens is None:
            tokens = torch.full((B, D), -1, dtype=torch.int32, device=dev)
        out = RoundsResult(tokens, torch.empty(B, dtype=torch.int32, device=dev),
                           torch.empty(B, R, dtype=torch.int32, device=dev))
    _req(out.tokens, "tokens", torch.int32, (B, D), dev)
    _req(out.n_revealed, "n_revealed", torch.int32, (B,), dev)
    _req(out.round_accepts, "round_accepts", torch.int32, (B, R), dev)
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(256, dev, sp)
    with torch.cuda.device(dev):
        rc = lib.spec_verify_anyorder_rounds(*_rounds_args(target_logits, draft_logits, order, revealed,
                                                           window, draft_tokens, u_accept, u_sample,
                                                           out, ws, sp))
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_anyorder_rounds")
    return out


def spec_anyorder_window(D: int, revealed: int, dtau: float) -> int:
    """W(i): the window of an outer step starting with `revealed` of D tokens
    revealed (cosine schedule, step dtau); computed by the library's host
    function."""
    return int(load().spec_anyorder_window(int(D), int(revealed), float(dtau)))


class PreparedCall:
    """A C-ABI call with every argument marshalled once.  Calling it issues
    exactly one library call (no tensor allocation, no checks) on the stream
    it was prepared for; the caller keeps the tensors alive."""

    def __init__(self, fn, args, keep, name):
        self._fn, self._args, self._keep, self.name = fn, args, keep, name

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc != SV_OK:
            raise SpecVerifyError(rc, self.name)


def prepare_dense(target_logits, draft_logits, draft_ids, u_accept, u_sample, out: VerifyResult,
                  stream: Optional[torch.cuda.Stream] = None) -> PreparedCall:
    """Validate once (by running the checked call) and return a PreparedCall
    that repeats spec_verify_dense on the same buffers."""
    spec_verify_dense(target_logits, draft_logits, draft_ids, u_accept, u_sample, out=out,
                      stream=stream)
    lib = load()
    dev = target_logits.device
    B, G1, V = target_logits.shape
    G = G1 - 1
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(workspace_size(B, G, V), dev, sp)
    args = (_ptr(target_logits), _ptr(draft_logits) if G > 0 else None,
            _logit_dtype(target_logits), _ptr(draft_ids), _ptr(u_accept), _ptr(u_sample), B, G, V,
            _ptr(out.n_accepted), _ptr(out.out_tokens), _ptr(out.residual), _ptr(out.accept_prob),
            ws.data_ptr(), ws.numel(), sp)
    keep = (target_logits, draft_logits, draft_ids, u_accept, u_sample, out, ws)
    return PreparedCall(lib.spec_verify_dense, args, keep, "spec_verify_dense")


def prepare_sparse(tgt_ids, tgt_probs, drf_ids, drf_probs, draft_tokens, u_accept, u_sample,
                   vocab_size, out: VerifyResult, stream=None) -> PreparedCall:
    spec_verify_sparse(tgt_ids, tgt_probs, drf_ids, drf_probs, draft_tokens, u_accept, u_sample,
                       vocab_size, out=out, stream=stream)
    lib = load()
    dev = tgt_ids.device
    B, G1, kt = tgt_ids.shape
    G = G1 - 1
    kd = drf_ids.shape[2] if drf_ids.dim() == 3 else 1
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(256, dev, sp)
    args = (_ptr(tgt_ids), _ptr(tgt_probs), kt, _ptr(drf_ids) if G else None,
            _ptr(drf_probs) if G else None, kd, _ptr(draft_tokens) if G else None,
            _ptr(u_accept) if G else None, _ptr(u_sample), B, G, int(vocab_size),
            _ptr(out.n_accepted), _ptr(out.out_tokens), _ptr(out.residual), _ptr(out.accept_prob),
            ws.data_ptr(), ws.numel(), sp)
    keep = (tgt_ids, tgt_probs, drf_ids, drf_probs, draft_tokens, u_accept, u_sample, out, ws)
    return PreparedCall(lib.spec_verify_sparse, args, keep, "spec_verify_sparse")


def prepare_anyorder(target_logits, draft_logits, order, draft_tokens, u_accept, u_sample,
                     out_tokens, stream=None) -> PreparedCall:
    res = spec_verify_anyorder(target_logits, draft_logits, order, draft_tokens, u_accept, u_sample,
                               out_tokens=out_tokens, stream=stream)
    lib = load()
    dev = target_logits.device
    B, D, V = target_logits.shape
    W = order.shape[1]
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(256, dev, sp)
    args = (_ptr(target_logits), _ptr(draft_logits), _logit_dtype(target_logits), _ptr(order),
            _ptr(draft_tokens), _ptr(u_accept), _ptr(u_sample), B, D, W, V, _ptr(res.n_accepted),
            _ptr(out_tokens), None, None, ws.data_ptr(), ws.numel(), sp)
    keep = (target_logits, draft_logits, order, draft_tokens, u_accept, u_sample, out_tokens, res, ws)
    return PreparedCall(lib.spec_verify_anyorder, args, keep, "spec_verify_anyorder")


def prepare_rounds(target_logits, draft_logits, order, revealed, window, draft_tokens, u_accept,
                   u_sample, out: RoundsResult,
                   stream: Optional[torch.cuda.Stream] = None) -> PreparedCall:
    """Validate once and return a PreparedCall repeating
    spec_verify_anyorder_rounds on the same buffers."""
    spec_verify_anyorder_rounds(target_logits, draft_logits, order, revealed, window, draft_tokens,
                                u_accept, u_sample, out=out, stream=stream)
    lib = load()
    dev = target_logits.device
    sp = _stream_ptr(stream, dev)
    ws = get_workspace(256, dev, sp)
    args = _rounds_args(target_logits, draft_logits, order, revealed, window, draft_tokens, u_accept,
                        u_sample, out, ws, sp)
    keep = (target_logits, draft_logits, order, revealed, window, draft_tokens, u_accept, u_sample,
            out, ws)
    return PreparedCall(lib.spec_verify_anyorder_rounds, args, keep, "spec_verify_anyorder_rounds")
