"""GB300-native verification step of speculative decoding.

A thin ctypes binding over ``libspecverify.so`` (C ABI in
``include/spec_verify.h``).  The functions take torch tensors on the GPU
and pass raw device pointers and the current CUDA stream; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback:
if the shared library is missing or cannot load, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libspecverify.so")

SPEC_F32 = 0
SPEC_BF16 = 1
SPEC_MAX_K = 32
SPEC_NO_BONUS = 1
SPEC_PREFER_RESIDENT = 2
SPEC_PREFER_STREAMING = 4
SPEC_PREFER_SPLIT = 8

SPEC_OK = 0
SPEC_ERR_NULL = -1
SPEC_ERR_SHAPE = -2
SPEC_ERR_DTYPE = -3
SPEC_ERR_K_TOO_LARGE = -4
SPEC_ERR_WORKSPACE = -5
SPEC_ERR_ALIGN = -6
SPEC_ERR_LAUNCH = -7
SPEC_ERR_DEVICE = -8
SPEC_ERR_STATIC_SCRATCH = -9
SPEC_STATIC_SCRATCH_BYTES = 8 << 20

SPEC_STATUS_BAD_TOKEN = 1
SPEC_STATUS_BAD_PARAM = 2
SPEC_STATUS_BAD_LOGITS = 4
SPEC_STATUS_BAD_K = 8
SPEC_STATUS_TIMEOUT = 16

EXPORTED = ("spec_workspace_bytes", "spec_verify_sample", "spec_verify_greedy", "spec_tv_budget",
            "spec_draft_confidence", "spec_verify_sample_static", "spec_status_string", "spec_set_wait_cycles")


class SpecArgs(ctypes.Structure):
    """Mirror of ``spec_args``."""

    _fields_ = [
        ("B", ctypes.c_int32),
        ("V", ctypes.c_int32),
        ("total_drafts", ctypes.c_int32),
        ("max_k", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("cu_draft", ctypes.c_void_p),
        ("target_logits", ctypes.c_void_p),
        ("ld_target", ctypes.c_int64),
        ("draft_logits", ctypes.c_void_p),
        ("ld_draft", ctypes.c_int64),
        ("draft_tokens", ctypes.c_void_p),
        ("cu_hist", ctypes.c_void_p),
        ("hist_tokens", ctypes.c_void_p),
        ("temperature", ctypes.c_void_p),
        ("rep_penalty", ctypes.c_void_p),
        ("top_p", ctypes.c_void_p),
        ("tv_budget", ctypes.c_void_p),
        ("uniforms", ctypes.c_void_p),
        ("flags", ctypes.c_uint32),
    ]


class SpecError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} ({code})")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libspecverify.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing; build it with "
                          f"`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    lib.spec_workspace_bytes.restype = ctypes.c_size_t
    lib.spec_workspace_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
    for name in ("spec_verify_sample", "spec_verify_greedy"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.POINTER(SpecArgs), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.spec_tv_budget.restype = ctypes.c_int
    lib.spec_tv_budget.argtypes = [ctypes.POINTER(SpecArgs), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.spec_draft_confidence.restype = ctypes.c_int
    lib.spec_draft_confidence.argtypes = [ctypes.POINTER(SpecArgs), ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.spec_verify_sample_static.restype = ctypes.c_int
    lib.spec_verify_sample_static.argtypes = [ctypes.POINTER(SpecArgs), ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p]
    lib.spec_status_string.restype = ctypes.c_char_p
    lib.spec_status_string.argtypes = [ctypes.c_int]
    lib.spec_set_wait_cycles.restype = ctypes.c_int64
    lib.spec_set_wait_cycles.argtypes = [ctypes.c_int64]
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().spec_status_string(int(code)).decode()


spec_status_string = status_string


def set_wait_cycles(cycles: int) -> int:
    """Bound (SM clock cycles) on every wait of the split-vocabulary kernel;
    <= 0 restores the default.  Returns the previous bound (a diagnostic
    hook: see ``spec_set_wait_cycles``)."""
    return int(load_library().spec_set_wait_cycles(int(cycles)))


spec_set_wait_cycles = set_wait_cycles


def spec_workspace_bytes(B: int, total_drafts: int, V: int) -> int:
    return int(load_library().spec_workspace_bytes(int(B), int(total_drafts), int(V)))


# ----------------------------------------------------------------- helpers

def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bf16 or fp32, got {t.dtype}")


def _stream_handle(stream) -> int:
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check_i32(name, t):
    import torch

    if t is not None and (t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")


def _check_f32(name, t):
    import torch

    if t is not None and (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous float32 CUDA tensor")


def make_args(*, target, cu_draft, draft_tokens, V: int, draft=None, cu_hist=None, hist=None,
              temperature=None, rep_penalty=None, top_p=None, tv_budget=None, uniforms=None,
              max_k: int = SPEC_MAX_K, flags: int = 0) -> SpecArgs:
    """Build ``spec_args`` from CUDA tensors.  Logit tensors are 2-D with a
    unit inner stride; their row stride is ``ld``."""
    for name, t in (("cu_draft", cu_draft), ("draft_tokens", draft_tokens), ("cu_hist", cu_hist),
                    ("hist", hist)):
        _check_i32(name, t)
    for name, t in (("temperature", temperature), ("rep_penalty", rep_penalty), ("top_p", top_p),
                    ("tv_budget", tv_budget), ("uniforms", uniforms)):
        _check_f32(name, t)
    if target.dim() != 2 or target.stride(1) != 1 or not target.is_cuda:
        raise TypeError("target logits must be a 2-D CUDA tensor with unit inner stride")
    a = SpecArgs()
    a.B = cu_draft.numel() - 1
    a.V = int(V)
    a.total_drafts = int(draft_tokens.numel()) if draft_tokens is not None else 0
    a.max_k = int(max_k)
    a.dtype = _dtype_code(target)
    a.cu_draft = _ptr(cu_draft)
    a.target_logits = _ptr(target)
    a.ld_target = target.stride(0)
    if draft is not None:
        if draft.dim() != 2 or draft.stride(1) != 1 or draft.dtype != target.dtype:
            raise TypeError("draft logits must match the target's dtype and be 2-D with unit inner stride")
        a.draft_logits = _ptr(draft)
        a.ld_draft = draft.stride(0)
    a.draft_tokens = _ptr(draft_tokens)
    a.cu_hist = _ptr(cu_hist)
    a.hist_tokens = _ptr(hist)
    a.temperature = _ptr(temperature)
    a.rep_penalty = _ptr(rep_penalty)
    a.top_p = _ptr(top_p)
    a.tv_budget = _ptr(tv_budget)
    a.uniforms = _ptr(uniforms)
    a.flags = int(flags)
    return a


def make_workspace(B: int, total_drafts: int, V: int, device="cuda"):
    import torch

    return torch.empty(max(spec_workspace_bytes(B, total_drafts, V), 256), dtype=torch.uint8, device=device)


def _outputs(args: SpecArgs, device, out_tokens, out_accepted, out_status):
    import torch

    n = args.total_drafts + args.B
    if out_tokens is None:
        out_tokens = torch.empty(n, dtype=torch.int32, device=device)
    if out_accepted is None:
        out_accepted = torch.empty(args.B, dtype=torch.int32, device=device)
    if out_status is None:
        out_status = torch.empty(args.B, dtype=torch.int32, device=device)
    return out_tokens, out_accepted, out_status


# ------------------------------------------------------------ entry points

def spec_verify_sample(args: SpecArgs, *, device=None, workspace=None, out_tokens=None, out_accepted=None,
                       out_status=None, stream=None):
    """Mentored speculative sampling through ``spec_verify_sample``.
    Returns (tokens [sum K + B], accepted [B], status [B]) CUDA int32 tensors."""
    import torch

    lib = load_library()
    device = device or torch.device("cuda", torch.cuda.current_device())
    if workspace is None:
        workspace = make_workspace(args.B, args.total_drafts, args.V, device)
    out_tokens, out_accepted, out_status = _outputs(args, device, out_tokens, out_accepted, out_status)
    rc = lib.spec_verify_sample(ctypes.byref(args), _ptr(out_tokens), _ptr(out_accepted), _ptr(out_status),
                                _ptr(workspace), workspace.numel(), _stream_handle(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_verify_sample")
    return out_tokens, out_accepted, out_status


def spec_verify_greedy(args: SpecArgs, *, device=None, workspace=None, out_tokens=None, out_accepted=None,
                       out_status=None, stream=None):
    """Greedy longest-prefix verification through ``spec_verify_greedy``."""
    import torch

    lib = load_library()
    device = device or torch.device("cuda", torch.cuda.current_device())
    if workspace is None:
        workspace = make_workspace(args.B, args.total_drafts, args.V, device)
    out_tokens, out_accepted, out_status = _outputs(args, device, out_tokens, out_accepted, out_status)
    rc = lib.spec_verify_greedy(ctypes.byref(args), _ptr(out_tokens), _ptr(out_accepted), _ptr(out_status),
                                _ptr(workspace), workspace.numel(), _stream_handle(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_verify_greedy")
    return out_tokens, out_accepted, out_status


def spec_draft_confidence(args: SpecArgs, threshold: float, *, device=None, workspace=None, stream=None):
    """Top-1 draft probability per draft row and the confidence-stopped draft
    count per request through ``spec_draft_confidence``.
    Returns (conf [sum K] float32, k_eff [B] int32, status [B] int32)."""
    import torch

    lib = load_library()
    device = device or torch.device("cuda", torch.cuda.current_device())
    if workspace is None:
        workspace = make_workspace(args.B, args.total_drafts, args.V, device)
    conf = torch.empty(max(args.total_drafts, 1), dtype=torch.float32, device=device)
    k_eff = torch.empty(args.B, dtype=torch.int32, device=device)
    status = torch.empty(args.B, dtype=torch.int32, device=device)
    rc = lib.spec_draft_confidence(ctypes.byref(args), float(threshold), _ptr(conf), _ptr(k_eff), _ptr(status),
                                   _ptr(workspace), workspace.numel(), _stream_handle(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_draft_confidence")
    return conf[:args.total_drafts], k_eff, status


def spec_verify_sample_static(args: SpecArgs, *, device=None, out_tokens=None, out_accepted=None, out_status=None,
                              stream=None):
    """``spec_verify_sample`` without a workspace, through
    ``spec_verify_sample_static``: the library's fixed per-device scratch
    (SPEC_STATIC_SCRATCH_BYTES) serves every call, so calls on one device
    must be ordered.  Pass preallocated outputs to allocate nothing here
    either."""
    import torch

    lib = load_library()
    device = device or torch.device("cuda", torch.cuda.current_device())
    out_tokens, out_accepted, out_status = _outputs(args, device, out_tokens, out_accepted, out_status)
    rc = lib.spec_verify_sample_static(ctypes.byref(args), _ptr(out_tokens), _ptr(out_accepted), _ptr(out_status),
                                       _stream_handle(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_verify_sample_static")
    return out_tokens, out_accepted, out_status


def spec_tv_budget(args: SpecArgs, *, device=None, workspace=None, stream=None, want_px: bool = True):
    """Per-position (tv, theta, p(x), q(x)) through ``spec_tv_budget``."""
    import torch

    lib = load_library()
    device = device or torch.device("cuda", torch.cuda.current_device())
    if workspace is None:
        workspace = make_workspace(args.B, args.total_drafts, args.V, device)
    n = max(args.total_drafts, 1)
    tv = torch.empty(n, dtype=torch.float32, device=device)
    theta = torch.empty(n, dtype=torch.float32, device=device)
    px = torch.empty(n, dtype=torch.float32, device=device) if want_px else None
    qx = torch.empty(n, dtype=torch.float32, device=device) if want_px else None
    rc = lib.spec_tv_budget(ctypes.byref(args), _ptr(tv), _ptr(theta), _ptr(px), _ptr(qx), _ptr(workspace),
                            workspace.numel(), _stream_handle(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_tv_budget")
    k = args.total_drafts
    return tv[:k], theta[:k], (px[:k] if px is not None else None), (qx[:k] if qx is not None else None)
