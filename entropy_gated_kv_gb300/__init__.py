"""EntropyCache denoising step on GB300: Python binding of the C ABI (include/entropycache.h).

Argument marshalling only: every stage of the step runs in the library's CUDA kernels.
PyTorch supplies device memory and streams. The library must be built in-tree first
(`python -m entropy_gated_kv_gb300.build`); importing the binding does not build it and
nothing here falls back to a CPU implementation.

Stages (EntropyCache, gist.science zh summary §2.2):
  entropy_decode     (a) softmax + greedy decode + Shannon entropy per candidate row
  select_recompute   (b)+(c) commit, max-entropy gate vs tau, decode history, recompute set
  kv_scatter         (c) fresh K/V rows of the recompute set into the cache
  partial_attention  (d) bidirectional attention of the recompute rows over all L rows
  step               all of the above for one denoising step over n layers
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import torch

from . import _capi as C
from ._capi import EcError  # noqa: F401

__all__ = [
    "Params",
    "DecodeState",
    "lib",
    "workspace",
    "entropy_decode",
    "entropy_decode_workspace_size",
    "entropy_decode_noalloc",
    "select_recompute",
    "candidates",
    "kv_scatter",
    "partial_attention",
    "partial_attention_workspace_size",
    "step",
    "step_workspace_size",
    "LayerWeights",
    "rope_table",
    "layer_forward",
    "layer_forward_workspace_size",
    "read_device_error",
    "EcError",
]


def lib() -> ctypes.CDLL:
    return C.load()


def _vp(t: torch.Tensor | None) -> ctypes.c_void_p | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("EntropyCache kernels take CUDA tensors (there is no CPU path)")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: torch.cuda.Stream | None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(d) -> int:
    if d in ("bf16", torch.bfloat16, C.EC_BF16):
        return C.EC_BF16
    if d in ("f32", torch.float32, C.EC_F32):
        return C.EC_F32
    raise ValueError(f"unsupported logits dtype {d!r}")


@dataclass
class Params:
    """Step shape and knobs (ec_params)."""

    B: int
    L: int
    Hq: int
    Hkv: int
    D: int
    V: int
    C_max: int
    k: int
    n_dec: int = 1
    tau: float = 1.0
    logits_dtype: object = "bf16"
    conf_threshold: float = 0.0  # > 0: commit only candidates at least this confident (at least one)
    scope_lo: int = 0  # the gate's scope [scope_lo, scope_hi) for block-by-block decoding;
    scope_hi: int = 0  # both 0: the whole sequence

    def c(self) -> C.EcParams:
        return C.EcParams(self.B, self.L, self.Hq, self.Hkv, self.D, self.V, self.C_max, self.k, self.n_dec,
                          float(self.tau), _dtype_code(self.logits_dtype), float(self.conf_threshold),
                          int(self.scope_lo), int(self.scope_hi))


class DecodeState:
    """Per-sequence decode state (ec_state) as CUDA tensors."""

    FIELDS = ("tokens", "mask", "ring", "ring_head", "ring_count", "dec_pos", "E", "flag", "idx", "R", "dev_err")

    def __init__(self, p: Params, device="cuda"):
        B, L, k = p.B, p.L, p.k
        z = lambda *s, dt=torch.int32: torch.zeros(*s, dtype=dt, device=device)  # noqa: E731
        self.tokens = z(B, L)
        self.mask = z(B, L, dt=torch.uint8)
        self.ring = z(B, k)
        self.ring_head = z(B)
        self.ring_count = z(B)
        self.dec_pos = z(B, p.n_dec)
        self.E = z(B, dt=torch.float32)
        self.flag = z(B, dt=torch.uint8)
        self.idx = z(B, L)
        self.R = z(B)
        self.dev_err = z(1)

    @classmethod
    def from_arrays(cls, p: Params, device="cuda", **arrays) -> "DecodeState":
        st = cls(p, device)
        for name, a in arrays.items():
            getattr(st, name).copy_(torch.as_tensor(a).to(getattr(st, name).dtype))
        return st

    def c(self) -> C.EcState:
        return C.EcState(*[_vp(getattr(self, f)) for f in self.FIELDS])

    def clone(self) -> "DecodeState":
        other = object.__new__(DecodeState)
        for f in self.FIELDS:
            setattr(other, f, getattr(self, f).clone())
        return other


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Scratch buffer for an entry point's workspace (the library needs no initial contents)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def entropy_decode_workspace_size(n_rows: int, V: int, dtype) -> int:
    return int(lib().ec_entropy_decode_workspace_size(n_rows, V, _dtype_code(dtype)))


def entropy_decode(logits: torch.Tensor, V: int | None = None, ws: torch.Tensor | None = None,
                   out: tuple | None = None, stream=None):
    """(a) ids int32, entropy fp32, log_conf fp32 for each row of logits [n_rows, row_stride]."""
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [n_rows, row_stride] with unit inner stride")
    n, V = logits.shape[0], (V if V is not None else logits.shape[1])
    code = _dtype_code(logits.dtype)
    if out is None:
        out = (torch.empty(n, dtype=torch.int32, device=logits.device),
               torch.empty(n, dtype=torch.float32, device=logits.device),
               torch.empty(n, dtype=torch.float32, device=logits.device))
    if ws is None:
        ws = workspace(entropy_decode_workspace_size(n, V, code), logits.device)
    st = lib().ec_entropy_decode(_vp(logits), logits.stride(0), n, V, code, _vp(out[0]), _vp(out[1]), _vp(out[2]),
                                 _vp(ws), ws.numel(), _stream(stream))
    C.check(st, "ec_entropy_decode")
    return out


def entropy_decode_noalloc(logits: torch.Tensor, V: int | None = None, out: tuple | None = None, stream=None):
    """(a) like entropy_decode, but with no workspace: for callers that cannot allocate device
    memory. The scratch is a 1 MiB array owned by the library; calls that overlap on the GPU
    race, and the first call on a device must come before any stream capture."""
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [n_rows, row_stride] with unit inner stride")
    n, V = logits.shape[0], (V if V is not None else logits.shape[1])
    code = _dtype_code(logits.dtype)
    if out is None:
        out = (torch.empty(n, dtype=torch.int32, device=logits.device),
               torch.empty(n, dtype=torch.float32, device=logits.device),
               torch.empty(n, dtype=torch.float32, device=logits.device))
    st = lib().ec_entropy_decode_noalloc(_vp(logits), logits.stride(0), n, V, code, _vp(out[0]), _vp(out[1]),
                                         _vp(out[2]), _stream(stream))
    C.check(st, "ec_entropy_decode_noalloc")
    return out


def lm_head_entropy_workspace_size(n_rows: int) -> int:
    return int(lib().ec_lm_head_entropy_workspace_size(n_rows))


def lm_head_entropy(hidden: torch.Tensor, weight: torch.Tensor, ws: torch.Tensor | None = None,
                    out: tuple | None = None, stream=None):
    """(a) from the hidden states: ids, entropy, log_conf of logits = hidden @ weight.T, which
    are computed on the tensor cores and never stored. hidden [n_rows, d_model] and weight
    [V, d_model]: contiguous CUDA bf16."""
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise ValueError("hidden and weight must be bf16")
    if hidden.dim() != 2 or weight.dim() != 2 or hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden [n_rows, d_model] and weight [V, d_model]")
    if not (hidden.is_contiguous() and weight.is_contiguous()):
        raise ValueError("hidden and weight must be contiguous")
    n, d = hidden.shape
    V = weight.shape[0]
    if out is None:
        out = (torch.empty(n, dtype=torch.int32, device=hidden.device),
               torch.empty(n, dtype=torch.float32, device=hidden.device),
               torch.empty(n, dtype=torch.float32, device=hidden.device))
    if ws is None:
        ws = workspace(lm_head_entropy_workspace_size(n), hidden.device)
    st = lib().ec_lm_head_entropy(_vp(hidden), _vp(weight), n, d, V, _vp(out[0]), _vp(out[1]), _vp(out[2]), _vp(ws),
                                  ws.numel(), _stream(stream))
    C.check(st, "ec_lm_head_entropy")
    return out


def select_recompute(p: Params, state: DecodeState, cand_pos, cand_count, ids, entropy, log_conf, stream=None):
    """(b)+(c) commit, gate, history push and recompute set; updates `state` in place."""
    pc, sc = p.c(), state.c()
    st = lib().ec_select_recompute(ctypes.byref(pc), ctypes.byref(sc), _vp(cand_pos), _vp(cand_count), _vp(ids),
                                   _vp(entropy), _vp(log_conf), _stream(stream))
    C.check(st, "ec_select_recompute")


def candidates(p: Params, state: DecodeState, mode: str, start: int, width: int, cand_pos=None, cand_count=None,
               stream=None):
    """Candidates of a block-wise ("block") or sliding-window ("sliding") decoding step: the
    masked positions of the window, built on the device from state.mask. Returns
    (cand_pos int32 [B, C_max], cand_count int32 [B])."""
    code = {"block": C.EC_CAND_BLOCK, "sliding": C.EC_CAND_SLIDING}[mode]
    dev = state.mask.device
    if cand_pos is None:
        cand_pos = torch.empty(p.B, p.C_max, dtype=torch.int32, device=dev)
    if cand_count is None:
        cand_count = torch.empty(p.B, dtype=torch.int32, device=dev)
    pc, sc = p.c(), state.c()
    st = lib().ec_candidates(ctypes.byref(pc), ctypes.byref(sc), code, int(start), int(width), _vp(cand_pos),
                             _vp(cand_count), _stream(stream))
    C.check(st, "ec_candidates")
    return cand_pos, cand_count


def kv_scatter(p: Params, k_cache, v_cache, k_new, v_new, idx, R, src_by_position: bool = False,
               dev_err=None, stream=None):
    """(c) k_cache[b, idx[b, r]] = k_new[b, r or idx[b, r]] (same for v) for r < R[b]."""
    pc = p.c()
    st = lib().ec_kv_scatter(ctypes.byref(pc), _vp(k_cache), _vp(v_cache), _vp(k_new), _vp(v_new),
                             int(bool(src_by_position)), _vp(idx), _vp(R), _vp(dev_err), _stream(stream))
    C.check(st, "ec_kv_scatter")


def partial_attention_workspace_size(p: Params) -> int:
    pc = p.c()
    return int(lib().ec_partial_attention_workspace_size(ctypes.byref(pc)))


def partial_attention(p: Params, q, k_cache, v_cache, R, out, scale: float | None = None,
                      ws: torch.Tensor | None = None, dev_err=None, stream=None):
    """(d) out[b, r, h] = softmax(scale q k^T) v over all L keys, for r < R[b]."""
    pc = p.c()
    if ws is None:
        ws = workspace(partial_attention_workspace_size(p), q.device)
    sc = (1.0 / math.sqrt(p.D)) if scale is None else float(scale)
    st = lib().ec_partial_attention(ctypes.byref(pc), _vp(q), _vp(k_cache), _vp(v_cache), _vp(R), sc, _vp(out),
                                    _vp(ws), ws.numel(), _vp(dev_err), _stream(stream))
    C.check(st, "ec_partial_attention")
    return out


def dense_attention(p: Params, q, k_cache, v_cache, out, scale: float | None = None, dev_err=None, stream=None):
    """(d) for a step known to be full: out[b, r, h] = softmax(scale q k^T) v over all L keys for
    every position r (q in position order), two query tiles per CTA with a softmax warpgroup
    each; D = 128."""
    pc = p.c()
    sc = (1.0 / math.sqrt(p.D)) if scale is None else float(scale)
    st = lib().ec_dense_attention(ctypes.byref(pc), _vp(q), _vp(k_cache), _vp(v_cache), sc, _vp(out), _vp(dev_err),
                                  _stream(stream))
    C.check(st, "ec_dense_attention")
    return out


@dataclass
class LayerWeights:
    """Weights of one LLaMA-style layer for layer_forward (ec_layer): CUDA bf16 tensors wq
    [Hq D, d], wk and wv [Hkv D, d], wo [d, Hq D], wg and wu [d_ff, d], wd [d, d_ff], gamma1 and
    gamma2 [d]; rope_cos and rope_sin fp32 [L, D / 2] (rope_table)."""

    wq: torch.Tensor
    wk: torch.Tensor
    wv: torch.Tensor
    wo: torch.Tensor
    wg: torch.Tensor
    wu: torch.Tensor
    wd: torch.Tensor
    gamma1: torch.Tensor
    gamma2: torch.Tensor
    rope_cos: torch.Tensor
    rope_sin: torch.Tensor
    eps: float = 1e-5

    @property
    def d_ff(self) -> int:
        return int(self.wg.shape[0])

    def c(self) -> C.EcLayer:
        return C.EcLayer(self.d_ff, float(self.eps), *[_vp(getattr(self, n)) for n in
                                                      ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "gamma1", "gamma2",
                                                       "rope_cos", "rope_sin")])


def rope_table(L: int, D: int, theta: float, device="cuda", stream=None):
    """RoPE cos / sin tables fp32 [L, D / 2] of the angles pos * theta^(-2i / D), built on the
    device in double precision (ec_rope_table)."""
    cs = torch.empty(L, D // 2, dtype=torch.float32, device=device)
    sn = torch.empty(L, D // 2, dtype=torch.float32, device=device)
    st = lib().ec_rope_table(int(L), int(D), float(theta), _vp(cs), _vp(sn), _stream(stream))
    C.check(st, "ec_rope_table")
    return cs, sn


def layer_forward_workspace_size(p: Params, d_ff: int) -> int:
    pc = p.c()
    return int(lib().ec_layer_forward_workspace_size(ctypes.byref(pc), int(d_ff)))


def layer_forward(p: Params, w: LayerWeights, idx, R, x_src, k_cache, v_cache, y=None, ws=None, dev_err=None,
                  stream=None):
    """The partial (R < L) or full forward of one layer for the recompute rows idx[b, :R[b]]
    (ec_layer_forward): refreshes k_cache / v_cache at those positions and returns y [B, L, d]
    (rows in recompute order, the first R[b] written)."""
    B, L, d = x_src.shape
    if y is None:
        y = torch.empty(B, L, d, dtype=torch.bfloat16, device=x_src.device)
    if ws is None:
        ws = workspace(layer_forward_workspace_size(p, w.d_ff), x_src.device)
    pc, wc = p.c(), w.c()
    st = lib().ec_layer_forward(ctypes.byref(pc), ctypes.byref(wc), _vp(idx), _vp(R), _vp(x_src), _vp(k_cache),
                                _vp(v_cache), _vp(y), _vp(ws), ws.numel(), _vp(dev_err), _stream(stream))
    C.check(st, "ec_layer_forward")
    return y


def step_workspace_size(p: Params) -> int:
    pc = p.c()
    return int(lib().ec_step_workspace_size(ctypes.byref(pc)))


def _ptr_array(ts) -> ctypes.Array:
    arr = (ctypes.c_void_p * max(1, len(ts)))()
    for i, t in enumerate(ts):
        arr[i] = t.data_ptr()
    return arr


def step(p: Params, state: DecodeState, logits, cand_pos, cand_count, layers: list[dict],
         scale: float | None = None, ws: torch.Tensor | None = None, stream=None):
    """One denoising step: (a)(b)(c) once, then scatter + attention for each layer.

    layers: dicts with k_cache, v_cache, k_src, v_src, q_src and out (CUDA bf16 tensors).
    """
    pc, sc = p.c(), state.c()
    if ws is None:
        ws = workspace(step_workspace_size(p), logits.device)
    names = ("k_cache", "v_cache", "k_src", "v_src", "q_src", "out")
    arrs = [_ptr_array([lay[n] for lay in layers]) for n in names]
    sc_ = (1.0 / math.sqrt(p.D)) if scale is None else float(scale)
    st = lib().ec_step(ctypes.byref(pc), ctypes.byref(sc), _vp(logits), _vp(cand_pos), _vp(cand_count), len(layers),
                       *arrs, sc_, _vp(ws), ws.numel(), _stream(stream))
    C.check(st, "ec_step")


def read_floor(buf: torch.Tensor, sink: torch.Tensor, stream=None) -> None:
    """A plain read of the whole buffer in the decode's launch shape (ec_read_floor): the floor
    for the decode's read of the same bytes. A measurement aid."""
    st = lib().ec_read_floor(_vp(buf), buf.numel() * buf.element_size(), _vp(sink), _stream(stream))
    C.check(st, "ec_read_floor")


def selftest_bounded_wait(dev_err: torch.Tensor, limit_ns: int, stream=None) -> None:
    """Runs the library's bounded wait on a barrier nothing completes; afterwards dev_err
    holds EC_DEVERR_TIMEOUT (read it with read_device_error)."""
    st = lib().ec_selftest_bounded_wait(_vp(dev_err), int(limit_ns), _stream(stream))
    C.check(st, "ec_selftest_bounded_wait")


def read_device_error(dev_err: torch.Tensor, stream=None) -> tuple[int, int]:
    """Synchronises the stream and returns (status, device error word)."""
    w = ctypes.c_int32(0)
    st = lib().ec_read_device_error(_vp(dev_err), ctypes.byref(w), _stream(stream))
    return int(st), int(w.value)
