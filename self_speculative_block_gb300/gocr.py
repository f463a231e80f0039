"""ctypes binding of libgocr.so (include/gocr.h): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels.  PyTorch
provides device memory (the allocator callback and the weight tensors) and the
CUDA stream; nothing here computes.  When the library has not been built the
import of a decoder fails loudly: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence

import numpy as np

from . import synth

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgocr.so")

GOCR_OK = 0
ERRORS = {-1: "EINVAL", -2: "ECAPACITY", -3: "ECUDA", -4: "EDEVICE", -5: "ETIMEOUT",
          -6: "ENOMEM", -7: "ESTATE"}
DTYPE_F32, DTYPE_BF16 = 0, 1
MODE_AR, MODE_SELFSPEC, MODE_DIFFUSION, MODE_REFINED = 0, 1, 2, 3
FWD_AR, FWD_DRAFT, FWD_VERIFY = 0, 1, 2
OPT_ATTENTION, OPT_ATTN_RANKS = 5, 6
TRACE_KERNELS, TRACE_CTAS = 1, 2
TRACE_CTA_SLOTS = 2048
ATTN_TCGEN05, ATTN_MMA_SYNC = 0, 1
MAX_BLOCK = 64
LAYER_TENSORS = 9

# every symbol include/gocr.h declares
EXPORTS = ("gocr_create", "gocr_prefill", "gocr_decode", "gocr_decode_batch", "gocr_decode_ex",
           "gocr_set_draft_override", "gocr_debug_forward", "gocr_debug_forward_batch", "gocr_read_kv", "gocr_get_state",
           "gocr_get_option", "gocr_read_trace", "gocr_last_error", "gocr_free",
           "gocr_op_linear_workspace", "gocr_op_linear", "gocr_op_linear_planes", "gocr_op_attention",
           "gocr_op_linear_static", "gocr_op_attention_ranges", "gocr_three_stream_ranges")


class GocrError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("max_ctx", ctypes.c_int32),
                ("max_block", ctypes.c_int32), ("max_requests", ctypes.c_int32),
                ("eos_id", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("mask_embed", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p), ("g_final", ctypes.c_void_p),
                ("layer", ctypes.POINTER(ctypes.c_void_p))]


class Stats(ctypes.Structure):
    _fields_ = [("rounds", ctypes.c_int64), ("forwards", ctypes.c_int64),
                ("committed", ctypes.c_int64), ("accepted_drafts", ctypes.c_int64),
                ("accept_hist", ctypes.c_int32 * (MAX_BLOCK + 1)), ("device_ms", ctypes.c_double)]

    def as_dict(self) -> dict:
        d = {k: getattr(self, k) for k in ("rounds", "forwards", "committed", "accepted_drafts",
                                           "device_ms")}
        d["accept_hist"] = list(self.accept_hist)
        d["tpf"] = self.committed / self.forwards if self.forwards else 0.0
        return d


class DecodeOpts(ctypes.Structure):
    _fields_ = [("tau", ctypes.c_float), ("draft_steps", ctypes.c_int32), ("temperature", ctypes.c_float),
                ("reserved", ctypes.c_uint32), ("seed", ctypes.c_uint64)]


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p)

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Open the library (built by __graft_entry__.build() or build.py)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libgocr.so is not built ({path}); run the package build first")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    P32 = ctypes.POINTER(ctypes.c_int32)
    sig = {
        "gocr_create": (i32, [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, ALLOC_FN, FREE_FN, vp,
                              ctypes.POINTER(vp)]),
        "gocr_prefill": (i32, [vp, i32, vp, i32]),
        "gocr_decode": (i32, [vp, i32, i32, i32, i32, P32, ctypes.POINTER(Stats)]),
        "gocr_decode_batch": (i32, [vp, i32, P32, i32, i32, P32, ctypes.POINTER(P32),
                                    ctypes.POINTER(Stats)]),
        "gocr_decode_ex": (i32, [vp, i32, P32, i32, i32, ctypes.POINTER(DecodeOpts), P32, ctypes.POINTER(P32),
                                 ctypes.POINTER(Stats)]),
        "gocr_set_draft_override": (i32, [vp, i32, P32, i32, P32, i32]),
        "gocr_debug_forward": (i32, [vp, i32, i32, P32, i32, ctypes.POINTER(ctypes.c_float)]),
        "gocr_debug_forward_batch": (i32, [vp, i32, P32, i32, P32, i32, ctypes.POINTER(ctypes.c_float)]),
        "gocr_read_kv": (i32, [vp, i32, i32, i32, i32, vp, vp]),
        "gocr_get_state": (i32, [vp, i32, P32, P32]),
        "gocr_read_trace": (i32, [vp, i32, vp, sz]),
        "gocr_get_option": (i32, [vp, i32, P32]),
        "gocr_last_error": (ctypes.c_char_p, [vp]),
        "gocr_free": (None, [vp]),
        "gocr_op_linear_workspace": (sz, [i32, i32, i32]),
        "gocr_op_linear": (i32, [i32, vp, vp, vp, i32, i32, i32, vp, sz, vp]),
        "gocr_op_linear_planes": (i32, [vp, vp, vp, vp, i32, i32, i32, vp, sz, ctypes.c_uint, vp]),
        "gocr_op_attention": (i32, [i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]),
        "gocr_op_linear_static": (i32, [i32, vp, vp, vp, i32, i32, i32, vp]),
        "gocr_op_attention_ranges": (i32, [i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]),
        "gocr_three_stream_ranges": (i32, [i32, i32, i32, P32, P32, P32, P32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def last_error(h=None) -> str:
    s = load().gocr_last_error(h)
    return s.decode() if s else ""


def _check(rc: int, h=None):
    if rc != GOCR_OK:
        raise GocrError(rc, last_error(h))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


# ----------------------------------------------------------------------------
# torch plumbing (device memory and streams only)
# ----------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def to_device(a: np.ndarray, dtype: str, device):
    """Host array (fp32 values, or bf16 bit patterns) -> device tensor in dtype."""
    torch = _torch()
    if dtype == synth.BF16:
        bits = a if a.dtype == np.uint16 else synth.bf16_bits(a)
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


class _TorchAllocator:
    """Device allocations for the library, served by torch's caching allocator."""

    def __init__(self, device):
        self.device = device
        self.live: Dict[int, object] = {}
        self.alloc_cb = ALLOC_FN(self._alloc)
        self.free_cb = FREE_FN(self._free)

    def _alloc(self, nbytes, _user):
        torch = _torch()
        try:
            t = torch.empty(int(nbytes), dtype=torch.uint8, device=self.device)
        except Exception:
            return None
        p = t.data_ptr()
        self.live[p] = t
        return p

    def _free(self, ptr, _user):
        self.live.pop(int(ptr or 0), None)


class Decoder:
    """One handle: a synthetic decoder resident on one GPU plus its KV caches."""

    def __init__(self, cfg: synth.ModelConfig, weights: dict, max_ctx: int, max_block: int = 32,
                 max_requests: int = 1, eos_id: int = -1, device: str = "cuda:0",
                 use_torch_alloc: bool = True):
        torch = _torch()
        self.lib = load()
        self.cfg = cfg
        self.device = torch.device(device)
        self.max_ctx, self.max_block, self.max_requests = max_ctx, max_block, max_requests
        dt = cfg.dtype
        with torch.cuda.device(self.device):
            self._keep: List[object] = []

            def up(a, d=dt):
                t = to_device(a, d, self.device)
                self._keep.append(t)
                return t.data_ptr()

            ptrs = []
            for lw in weights["layers"]:
                for name in synth.LAYER_MATS:
                    ptrs.append(up(lw[name]))
                ptrs.append(up(lw["g_attn"], synth.F32))
                ptrs.append(up(lw["g_mlp"], synth.F32))
            self._layer_ptrs = (ctypes.c_void_p * len(ptrs))(*ptrs)
            w = Weights(up(weights["embed"]), up(weights["mask_embed"]), up(weights["lm_head"]),
                        up(weights["g_final"], synth.F32),
                        ctypes.cast(self._layer_ptrs, ctypes.POINTER(ctypes.c_void_p)))
            c = Config(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn,
                       cfg.vocab, DTYPE_BF16 if dt == synth.BF16 else DTYPE_F32, cfg.rms_eps,
                       cfg.rope_theta, max_ctx, max_block, max_requests, eos_id)
            self._alloc = _TorchAllocator(self.device) if use_torch_alloc else None
            h = ctypes.c_void_p()
            stream = torch.cuda.current_stream(self.device).cuda_stream
            rc = self.lib.gocr_create(ctypes.byref(c), ctypes.byref(w), stream,
                                      self._alloc.alloc_cb if self._alloc else ALLOC_FN(),
                                      self._alloc.free_cb if self._alloc else FREE_FN(), None,
                                      ctypes.byref(h))
            _check(rc, None)
            self.h = h

    # ------------------------------------------------------------------ calls
    def close(self):
        if getattr(self, "h", None):
            self.lib.gocr_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, req: int, prefix) -> None:
        """prefix: host array [P, hidden] (values of cfg.dtype) or a device tensor."""
        torch = _torch()
        if isinstance(prefix, np.ndarray):
            if self.cfg.dtype == synth.BF16:
                host = np.ascontiguousarray(prefix if prefix.dtype == np.uint16 else synth.bf16_bits(prefix))
            else:
                host = np.ascontiguousarray(prefix, dtype=np.float32)
            _check(self.lib.gocr_prefill(self.h, req, host.ctypes.data, host.shape[0]), self.h)
        else:
            assert isinstance(prefix, torch.Tensor) and prefix.is_contiguous()
            _check(self.lib.gocr_prefill(self.h, req, prefix.data_ptr(), prefix.shape[0]), self.h)

    def decode(self, req: int, mode: int, B: int, max_new: int, out: Optional[np.ndarray] = None):
        out = np.zeros(max_new, np.int32) if out is None else out
        st = Stats()
        _check(self.lib.gocr_decode(self.h, req, mode, B, max_new, _p32(out), ctypes.byref(st)), self.h)
        return out, st.as_dict()

    def decode_batch(self, reqs: Sequence[int], mode: int, B: int, max_new: Sequence[int]):
        n = len(reqs)
        r = _i32(reqs)
        mn = _i32(max_new)
        outs = [np.zeros(int(m), np.int32) for m in max_new]
        optr = (ctypes.POINTER(ctypes.c_int32) * n)(*[_p32(o) for o in outs])
        sts = (Stats * n)()
        _check(self.lib.gocr_decode_batch(self.h, n, _p32(r), mode, B, _p32(mn), optr, sts), self.h)
        return outs, [s.as_dict() for s in sts]

    def decode_ex(self, reqs: Sequence[int], mode: int, B: int, max_new: Sequence[int], tau: float = 0.0,
                  draft_steps: int = 1, temperature: float = 0.0, seed: int = 0):
        """Any decode mode over several requests; MODE_DIFFUSION takes the
        confidence threshold tau, MODE_REFINED the draft-side threshold tau and
        at most draft_steps draft forwards per round; MODE_AR and MODE_SELFSPEC
        sample at temperature > 0 with the random-number key seed."""
        n = len(reqs)
        r = _i32(reqs)
        mn = _i32(max_new)
        outs = [np.zeros(int(m), np.int32) for m in max_new]
        optr = (ctypes.POINTER(ctypes.c_int32) * n)(*[_p32(o) for o in outs])
        sts = (Stats * n)()
        opts = DecodeOpts(float(tau), int(draft_steps), float(temperature), 0, int(seed))
        _check(self.lib.gocr_decode_ex(self.h, n, _p32(r), mode, B, ctypes.byref(opts), _p32(mn), optr, sts),
               self.h)
        return outs, [s.as_dict() for s in sts]

    def set_draft_override(self, req: int, ref: Sequence[int], schedule: Sequence[int]):
        ref_a = _i32(ref)
        sch = _i32(schedule)
        _check(self.lib.gocr_set_draft_override(self.h, req, _p32(ref_a), len(ref_a), _p32(sch),
                                                len(sch)), self.h)

    def clear_draft_override(self, req: int):
        z = np.zeros(1, np.int32)
        _check(self.lib.gocr_set_draft_override(self.h, req, _p32(z), 0, _p32(z), 0), self.h)

    def debug_forward(self, req: int, kind: int, tokens: Sequence[int]) -> np.ndarray:
        t = _i32(tokens)
        logits = np.zeros((len(t), self.cfg.vocab), np.float32)
        _check(self.lib.gocr_debug_forward(self.h, req, kind, _p32(t), len(t),
                                           logits.ctypes.data_as(ctypes.POINTER(ctypes.c_float))),
               self.h)
        return logits

    def debug_forward_batch(self, reqs: Sequence[int], kind: int, tokens) -> np.ndarray:
        """One batched forward over several requests; tokens [n_req, n]; logits [n_req, n, vocab]."""
        r = _i32(reqs)
        t = _i32(tokens)
        n_req, n = t.shape
        logits = np.zeros((n_req, n, self.cfg.vocab), np.float32)
        _check(self.lib.gocr_debug_forward_batch(self.h, n_req, _p32(r), kind, _p32(t.reshape(-1)), n,
                                                 logits.ctypes.data_as(ctypes.POINTER(ctypes.c_float))), self.h)
        return logits

    def read_kv(self, req: int, layer: int, pos0: int, n: int):
        """Cached K (rotated) and V of positions pos0..pos0+n-1: two fp32 arrays [n, Hkv, d]."""
        shape = (n, self.cfg.n_kv_heads, self.cfg.head_dim)
        k = np.zeros(shape, np.float32)
        v = np.zeros(shape, np.float32)
        _check(self.lib.gocr_read_kv(self.h, req, layer, pos0, n, k.ctypes.data, v.ctypes.data), self.h)
        return k, v

    def attention_kind(self) -> int:
        """ATTN_TCGEN05 or ATTN_MMA_SYNC, fixed at create time (by chunks per rank, or GOCR_ATTN=tc | mma)."""
        return self._option(OPT_ATTENTION)

    def attention_ranks(self) -> int:
        """Key-chunk ranks of the handle's attention (fixed at create time)."""
        return self._option(OPT_ATTN_RANKS)

    def _option(self, opt: int) -> int:
        v = ctypes.c_int32()
        _check(self.lib.gocr_get_option(self.h, opt, ctypes.byref(v)), self.h)
        return v.value

    def read_kernel_trace(self) -> np.ndarray:
        """Per-launch timeline of the last debug forward run with one kernel per
        operation: uint64 [5 L + 1, 8] (first start, first and last dependency
        release, last end, last mainloop end, last split-K exchange end; ns)."""
        out = np.zeros((5 * self.cfg.n_layers + 1, 8), np.uint64)
        _check(self.lib.gocr_read_trace(self.h, TRACE_KERNELS, out.ctypes.data, out.size), self.h)
        return out

    def read_cta_trace(self) -> np.ndarray:
        """Per-CTA timelines of the last debug forward (GOCR_OP_TRACE=2 at
        create): uint64 [5 L + 1, 2048, 8]; CTA c of a launch in slot c, the
        attention merge kernel's CTAs from slot 1024; zero where unreached."""
        out = np.zeros((5 * self.cfg.n_layers + 1, TRACE_CTA_SLOTS, 8), np.uint64)
        _check(self.lib.gocr_read_trace(self.h, TRACE_CTAS, out.ctypes.data, out.size), self.h)
        return out

    def state(self, req: int):
        cl = ctypes.c_int32()
        x0 = ctypes.c_int32()
        _check(self.lib.gocr_get_state(self.h, req, ctypes.byref(cl), ctypes.byref(x0)), self.h)
        return cl.value, x0.value


# ----------------------------------------------------------------------------
# single-kernel calls on torch tensors
# ----------------------------------------------------------------------------

def _dt(t) -> int:
    torch = _torch()
    return DTYPE_BF16 if t.dtype == torch.bfloat16 else DTYPE_F32


def op_linear(x, w, workspace=None):
    """y[T, N] fp32 = x[T, K] w[N, K]^T through the decoder's split-K GEMM."""
    torch = _torch()
    lib = load()
    T, K = x.shape
    N = w.shape[0]
    y = torch.empty((T, N), dtype=torch.float32, device=x.device)
    need = lib.gocr_op_linear_workspace(T, N, K)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    _check(lib.gocr_op_linear(_dt(x), x.data_ptr(), w.data_ptr(), y.data_ptr(), T, N, K,
                              workspace.data_ptr(), workspace.numel(), stream))
    return y


OP_OVERLAP = 1


def op_linear_planes(x_hi, x_lo, w, workspace=None, flags: int = 0):
    """y[T, N] fp32 = (x_hi + x_lo)[T, K] w[N, K]^T on bf16 planes, the
    decoder's GEMM on its activation planes.  flags=OP_OVERLAP launches it as
    the decoder does (programmatic dependent launch; w must not be written by
    the stream's previous kernel)."""
    torch = _torch()
    lib = load()
    T, K = x_hi.shape
    N = w.shape[0]
    if x_lo.shape != x_hi.shape or not (x_hi.dtype == x_lo.dtype == w.dtype == torch.bfloat16):
        raise ValueError("op_linear_planes takes bf16 planes of one shape and bf16 weights")
    y = torch.empty((T, N), dtype=torch.float32, device=x_hi.device)
    need = lib.gocr_op_linear_workspace(T, N, K)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=x_hi.device)
    stream = torch.cuda.current_stream(x_hi.device).cuda_stream
    _check(lib.gocr_op_linear_planes(x_hi.data_ptr(), x_lo.data_ptr(), w.data_ptr(), y.data_ptr(), T, N, K,
                                     workspace.data_ptr(), workspace.numel(), flags, stream))
    return y


def op_linear_static(x, w):
    """op_linear without a workspace: the library's static device scratch array
    (for callers that cannot allocate device memory)."""
    torch = _torch()
    lib = load()
    T, K = x.shape
    N = w.shape[0]
    y = torch.empty((T, N), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):  # the library takes the scratch address of the current device
        stream = torch.cuda.current_stream(x.device).cuda_stream
        _check(lib.gocr_op_linear_static(_dt(x), x.data_ptr(), w.data_ptr(), y.data_ptr(), T, N, K, stream))
    return y


def three_stream_ranges(P: int, N: int, B: int):
    """Row key intervals (lim, lo2, hi2) and rotary positions of the joint
    training mask over [prefix, clean, corrupted 1, corrupted 2] (host int32
    arrays of P + 3 N), from the library."""
    n = P + 3 * N
    lim, lo2, hi2, pos = (np.zeros(n, np.int32) for _ in range(4))
    _check(load().gocr_three_stream_ranges(P, N, B, _p32(lim), _p32(lo2), _p32(hi2), _p32(pos)))
    return lim, lo2, hi2, pos


def op_attention(q, kc, vc, lim, dtype: int, lo2=None, hi2=None):
    """The decoder's attention kernel for `dtype` (DTYPE_BF16 / DTYPE_F32).

    q [T, Hq, d], kc and vc [Hkv, cap, d]: fp32 tensors for DTYPE_F32, or
    (hi, lo) pairs of bf16 tensors for DTYPE_BF16; lim int32 [T] on the
    device; lo2, hi2 (optional) int32 [T] on the device: a second key
    interval per row.  Returns fp32 [T, Hq, d]."""
    torch = _torch()
    lib = load()
    pair = lambda t: (t[0], t[1]) if isinstance(t, (tuple, list)) else (t, None)
    (qh, ql), (kh, kl), (vh, vl) = pair(q), pair(kc), pair(vc)
    T, Hq, d = qh.shape
    Hkv, cap, _ = kh.shape
    o = torch.empty((T, Hq, d), dtype=torch.float32, device=qh.device)
    ptr = lambda t: t.data_ptr() if t is not None else None
    stream = torch.cuda.current_stream(qh.device).cuda_stream
    _check(lib.gocr_op_attention_ranges(dtype, ptr(qh), ptr(ql), ptr(kh), ptr(kl), ptr(vh), ptr(vl), o.data_ptr(),
                                        lim.data_ptr(), ptr(lo2), ptr(hi2), T, Hq, Hkv, d, cap, stream))
    return o
