"""ctypes declarations of the EntropyCache C ABI (include/entropycache.h).

Loading fails loudly when the in-tree library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "libentropycache.so"

EC_OK = 0
EC_ERR_INVALID_ARG = 1
EC_ERR_UNSUPPORTED = 2
EC_ERR_CUDA = 3
EC_ERR_DEVICE_CHECK = 4
EC_ERR_TIMEOUT = 5

EC_DEVERR_BAD_CAND_POS = 0x1
EC_DEVERR_BAD_IDX = 0x2
EC_DEVERR_BAD_R = 0x4
EC_DEVERR_TIMEOUT = 0x8

EC_F32 = 0
EC_BF16 = 1

EC_CAND_BLOCK = 0
EC_CAND_SLIDING = 1

EC_NOALLOC_SCRATCH_BYTES = 1 << 20

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_f32 = ctypes.c_float


class EcParams(ctypes.Structure):
    _fields_ = [
        ("B", _i32), ("L", _i32), ("Hq", _i32), ("Hkv", _i32), ("D", _i32), ("V", _i32),
        ("C_max", _i32), ("k", _i32), ("n_dec", _i32), ("tau", _f32), ("logits_dtype", _i32),
        ("conf_threshold", _f32), ("scope_lo", _i32), ("scope_hi", _i32),
    ]


class EcState(ctypes.Structure):
    _fields_ = [
        ("tokens", _p), ("mask", _p), ("ring", _p), ("ring_head", _p), ("ring_count", _p),
        ("dec_pos", _p), ("E", _p), ("flag", _p), ("idx", _p), ("R", _p), ("dev_err", _p),
    ]


class EcLayer(ctypes.Structure):
    _fields_ = [
        ("d_ff", _i32), ("eps", _f32), ("wq", _p), ("wk", _p), ("wv", _p), ("wo", _p), ("wg", _p), ("wu", _p),
        ("wd", _p), ("gamma1", _p), ("gamma2", _p), ("rope_cos", _p), ("rope_sin", _p),
    ]


# name -> (restype, argtypes)
SIGNATURES: dict[str, tuple] = {
    "ec_status_string": (ctypes.c_char_p, [_i32]),
    "ec_version": (_i32, []),
    "ec_read_device_error": (_i32, [_p, ctypes.POINTER(_i32), _p]),
    "ec_entropy_decode_workspace_size": (_sz, [_i32, _i32, _i32]),
    "ec_entropy_decode": (_i32, [_p, _i64, _i32, _i32, _i32, _p, _p, _p, _p, _sz, _p]),
    "ec_entropy_decode_noalloc": (_i32, [_p, _i64, _i32, _i32, _i32, _p, _p, _p, _p]),
    "ec_selftest_bounded_wait": (_i32, [_p, ctypes.c_uint64, _p]),
    "ec_candidates": (_i32, [_p, _p, _i32, _i32, _i32, _p, _p, _p]),
    "ec_layer_forward_workspace_size": (_sz, [_p, _i32]),
    "ec_layer_forward": (_i32, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p, _p]),
    "ec_rope_table": (_i32, [_i32, _i32, _f32, _p, _p, _p]),
    "ec_read_floor": (_i32, [_p, _sz, _p, _p]),
    "ec_lm_head_entropy_workspace_size": (_sz, [_i32]),
    "ec_lm_head_entropy": (_i32, [_p, _p, _i32, _i32, _i32, _p, _p, _p, _p, _sz, _p]),
    "ec_select_recompute": (_i32, [ctypes.POINTER(EcParams), ctypes.POINTER(EcState), _p, _p, _p, _p, _p, _p]),
    "ec_kv_scatter": (_i32, [ctypes.POINTER(EcParams), _p, _p, _p, _p, _i32, _p, _p, _p, _p]),
    "ec_partial_attention_workspace_size": (_sz, [ctypes.POINTER(EcParams)]),
    "ec_partial_attention": (_i32, [ctypes.POINTER(EcParams), _p, _p, _p, _p, _f32, _p, _p, _sz, _p, _p]),
    "ec_dense_attention": (_i32, [ctypes.POINTER(EcParams), _p, _p, _p, _f32, _p, _p, _p]),
    "ec_step_workspace_size": (_sz, [ctypes.POINTER(EcParams)]),
    "ec_step": (_i32, [ctypes.POINTER(EcParams), ctypes.POINTER(EcState), _p, _p, _p, _i32,
                       ctypes.POINTER(_p), ctypes.POINTER(_p), ctypes.POINTER(_p), ctypes.POINTER(_p),
                       ctypes.POINTER(_p), ctypes.POINTER(_p), _f32, _p, _sz, _p]),
}

_LIB: ctypes.CDLL | None = None


def load(path: Path | str | None = None) -> ctypes.CDLL:
    """Loads the in-tree library (once) and declares every entry point."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = Path(path) if path is not None else LIB_PATH
    if not p.exists():
        raise ImportError(
            f"{p} is missing: build the EntropyCache CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()'); there is no CPU fallback")
    lib = ctypes.CDLL(str(p))
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


class EcError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = load().ec_status_string(status).decode()
        super().__init__(f"{what} failed: {name} ({status})")


def check(status: int, what: str) -> None:
    if status != EC_OK:
        raise EcError(status, what)
