"""Thin ctypes binding of libdr (include/dr.h), argument marshalling only.

Each ``dr_*`` function here has the name and argument order of the C entry
point and returns its status code; every computation happens in the CUDA
library.  Tensor arguments may be ``torch.Tensor`` (their ``data_ptr()`` is
passed), plain integer addresses, or ``None`` (NULL).  ``stream`` is a
``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or ``None`` for the
current torch stream.

Importing this module loads ``libdr.so`` from the package directory and fails
loudly if it has not been built (``__graft_entry__.build()`` or
``python -m recurrent_associative_memory_gb300.build``).  There is no fallback
path of any kind.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int, c_size_t, c_void_p, c_char_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdr.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libdr.so is not built at {LIB_PATH}; run "
                      "`python -m recurrent_associative_memory_gb300.build` (needs nvcc)")
_lib = ctypes.CDLL(LIB_PATH)

DR_GDN, DR_KLA, DR_PGDN, DR_KDN, DR_KDA, DR_PKDA, DR_IKDN, DR_EKDN = 0, 1, 2, 3, 4, 5, 6, 7
VARIANT_IDS = {"gdn": DR_GDN, "kla": DR_KLA, "pgdn": DR_PGDN, "kdn": DR_KDN, "kda": DR_KDA,
               "pkda": DR_PKDA, "ikdn": DR_IKDN, "ekdn": DR_EKDN}
DR_FP32, DR_BF16 = 0, 1
STATUS = {0: "DR_OK", -1: "DR_ERR_NULL", -2: "DR_ERR_SHAPE", -3: "DR_ERR_DTYPE",
          -4: "DR_ERR_ALIGN", -5: "DR_ERR_WORKSPACE", -6: "DR_ERR_CUDA", -7: "DR_ERR_TIMEOUT",
          -8: "DR_ERR_NONFINITE", -9: "DR_ERR_UNSUPPORTED", -10: "DR_ERR_ARG"}
globals().update({name: code for code, name in STATUS.items()})


class DrParams(ctypes.Structure):
    """Mirror of ``dr_params`` (field order and types as in include/dr.h)."""
    _fields_ = [
        ("dtype", c_int), ("q_l2norm", c_int), ("k_l2norm", c_int),
        ("eta", c_void_p), ("alphaP", c_void_p), ("betaP", c_void_p), ("mu", c_void_p),
        ("x", c_float), ("log_floor", c_float),
        ("omega", c_void_p), ("r", c_void_p), ("info_scale", c_float),
        ("aux_init", c_void_p), ("aux_final", c_void_p),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
        ("check_finite", c_int),
    ]


_lib.dr_params_init.argtypes = [ctypes.POINTER(DrParams)]
_lib.dr_params_init.restype = None
_lib.dr_chunk_fwd.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, ctypes.POINTER(DrParams),
                              c_int, c_float, c_void_p, c_void_p, c_void_p,
                              c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]
_lib.dr_chunk_fwd.restype = c_int
_lib.dr_decode_step.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, ctypes.POINTER(DrParams),
                                c_int, c_float, c_void_p, c_void_p, c_void_p,
                                c_int, c_int, c_int, c_int, c_void_p]
_lib.dr_decode_step.restype = c_int
_lib.dr_chunk_fwd_workspace_bytes.argtypes = [c_int] * 8
_lib.dr_chunk_fwd_workspace_bytes.restype = c_size_t
_lib.dr_get_device_status.argtypes = [c_void_p]
_lib.dr_get_device_status.restype = c_int
_lib.dr_status_string.argtypes = [c_int]
_lib.dr_status_string.restype = c_char_p
_lib.dr_chunk_fwd_path.argtypes = [c_int] * 5
_lib.dr_chunk_fwd_path.restype = c_char_p
_lib.dr_chunk_fwd_noalloc.argtypes = _lib.dr_chunk_fwd.argtypes
_lib.dr_chunk_fwd_noalloc.restype = c_int


class DrGrads(ctypes.Structure):
    """Mirror of dr_grads (include/dr.h): device pointers of the backward's outputs."""
    _fields_ = [("dq", c_void_p), ("dk", c_void_p), ("dv", c_void_p), ("d_log_alpha", c_void_p),
                ("d_eta", c_void_p), ("d_init_state", c_void_p), ("d_alphaP", c_void_p),
                ("d_betaP", c_void_p), ("d_mu", c_void_p), ("d_aux_init", c_void_p),
                ("d_aux_final", c_void_p), ("d_omega", c_void_p), ("d_r", c_void_p)]


_lib.dr_chunk_bwd.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, ctypes.POINTER(DrParams),
                             c_int, ctypes.c_float, c_void_p, c_void_p, c_void_p,
                             ctypes.POINTER(DrGrads), c_int, c_int, c_int, c_int, c_int, c_int,
                             c_void_p]
_lib.dr_chunk_bwd.restype = c_int
_lib.dr_chunk_bwd_workspace_bytes.argtypes = [c_int] * 8
_lib.dr_chunk_bwd_workspace_bytes.restype = c_size_t
_lib.dr_set_chain_fault_for_testing.argtypes = [ctypes.c_longlong, ctypes.c_ulonglong]
_lib.dr_set_chain_fault_for_testing.restype = c_int

# size of the library-owned scratch behind dr_chunk_fwd_noalloc (include/dr.h)
DR_NOALLOC_SCRATCH_BYTES = 64 << 20


class DrError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({dr_status_string(status)})")


def check(status: int, where: str = "libdr") -> None:
    """Raise DrError for a non-zero status."""
    if status != 0:
        raise DrError(status, where)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def dr_params_init() -> DrParams:
    p = DrParams()
    _lib.dr_params_init(ctypes.byref(p))
    return p


def make_params(dtype=DR_BF16, q_l2norm=False, k_l2norm=False, eta=None, alphaP=None,
                betaP=None, mu=None, x=1.5, log_floor=1e-12, omega=None, r=None,
                info_scale=1.0, aux_init=None, aux_final=None, workspace=None,
                workspace_bytes=0, check_finite=False) -> DrParams:
    """Fill a DrParams from tensors/addresses (marshalling only)."""
    p = dr_params_init()
    p.dtype = int(dtype)
    p.q_l2norm, p.k_l2norm = int(bool(q_l2norm)), int(bool(k_l2norm))
    p.eta, p.alphaP, p.betaP, p.mu = _ptr(eta), _ptr(alphaP), _ptr(betaP), _ptr(mu)
    p.x, p.log_floor = float(x), float(log_floor)
    p.omega, p.r, p.info_scale = _ptr(omega), _ptr(r), float(info_scale)
    p.aux_init, p.aux_final = _ptr(aux_init), _ptr(aux_final)
    p.workspace, p.workspace_bytes = _ptr(workspace), int(workspace_bytes)
    p.check_finite = int(bool(check_finite))
    return p


def dr_chunk_fwd(q, k, v, log_alpha, params: DrParams, variant: int, eps: float, init_state,
                 out, final_state, B: int, T: int, H: int, dk: int, dv: int, chunk: int,
                 stream=None) -> int:
    return _lib.dr_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), ctypes.byref(params),
                             int(variant), float(eps), _ptr(init_state), _ptr(out),
                             _ptr(final_state), B, T, H, dk, dv, chunk, _stream(stream))


def dr_decode_step(q, k, v, log_alpha, params: DrParams, variant: int, eps: float, state,
                   aux_state, out, B: int, H: int, dk: int, dv: int, stream=None) -> int:
    return _lib.dr_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), ctypes.byref(params),
                               int(variant), float(eps), _ptr(state), _ptr(aux_state), _ptr(out),
                               B, H, dk, dv, _stream(stream))


def dr_chunk_fwd_workspace_bytes(variant, dtype, B, T, H, dk, dv, chunk) -> int:
    return _lib.dr_chunk_fwd_workspace_bytes(variant, dtype, B, T, H, dk, dv, chunk)


def dr_get_device_status(stream=None) -> int:
    return _lib.dr_get_device_status(_stream(stream))


def dr_status_string(status: int) -> str:
    return _lib.dr_status_string(int(status)).decode()


def dr_chunk_fwd_path(variant, dtype, dk, dv, chunk) -> str:
    return _lib.dr_chunk_fwd_path(variant, dtype, dk, dv, chunk).decode()


def dr_chunk_fwd_noalloc(q, k, v, log_alpha, params: DrParams, variant: int, eps: float,
                         init_state, out, final_state, B: int, T: int, H: int, dk: int, dv: int,
                         chunk: int, stream=None) -> int:
    return _lib.dr_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                     ctypes.byref(params), int(variant), float(eps),
                                     _ptr(init_state), _ptr(out), _ptr(final_state), B, T, H, dk,
                                     dv, chunk, _stream(stream))


def dr_set_chain_fault_for_testing(withhold_flag: int, wait_ns: int) -> int:
    """Test only: withhold one hand-over flag of the chained prep and set the wait limit."""
    return _lib.dr_set_chain_fault_for_testing(int(withhold_flag), int(wait_ns))


def make_grads(**ptrs) -> DrGrads:
    """A dr_grads with the given fields set (tensors or raw addresses; others NULL)."""
    g = DrGrads()
    for name, value in ptrs.items():
        setattr(g, name, _ptr(value))
    return g


def dr_chunk_bwd(q, k, v, log_alpha, params: DrParams, variant: int, eps: float, init_state,
                 d_out, d_final_state, grads: DrGrads, B: int, T: int, H: int, dk: int, dv: int,
                 chunk: int, stream=None) -> int:
    return _lib.dr_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), ctypes.byref(params),
                             int(variant), float(eps), _ptr(init_state), _ptr(d_out),
                             _ptr(d_final_state), ctypes.byref(grads), B, T, H, dk, dv, chunk,
                             _stream(stream))


def dr_chunk_bwd_workspace_bytes(variant, dtype, B, T, H, dk, dv, chunk) -> int:
    return _lib.dr_chunk_bwd_workspace_bytes(variant, dtype, B, T, H, dk, dv, chunk)
