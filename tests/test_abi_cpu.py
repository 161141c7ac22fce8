"""Host-side checks of the C-ABI library (no GPU needed, no kernel launched).

* libdr.so exports every function include/dr.h declares;
* the ctypes mirror of dr_params has the C compiler's layout;
* argument validation rejects bad calls before anything reaches CUDA.  Every
  call here fails validation, so no fake pointer is ever dereferenced.
"""

import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dr.h")
LIB = os.path.join(ROOT, "recurrent_associative_memory_gb300", "libdr.so")


@pytest.fixture(scope="module")
def dr():
    if not os.path.exists(LIB):
        from recurrent_associative_memory_gb300 import build
        build.build()
    from recurrent_associative_memory_gb300 import dr as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dr_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("dr_chunk_fwd", "dr_decode_step", "dr_chunk_fwd_workspace_bytes",
              "dr_get_device_status", "dr_status_string", "dr_params_init"):
        assert n in names


def test_library_exports_every_declared_symbol(dr):
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (dr_[a-z0-9_]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(LIB)
    for n in declared_functions():
        assert hasattr(lib, n)


def test_params_struct_layout_matches_c(dr):
    fields = [f for f, _ in dr.DrParams._fields_]
    src = "#include <stdio.h>\n#include <stddef.h>\n#include \"dr.h\"\nint main(void){\n"
    src += 'printf("%zu\\n", sizeof(dr_params));\n'
    for f in fields:
        src += f'printf("%zu\\n", offsetof(dr_params, {f}));\n'
    src += "return 0;}\n"
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "layout.c")
        exe = os.path.join(td, "layout")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
        vals = [int(x) for x in subprocess.run([exe], capture_output=True, text=True,
                                               check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(dr.DrParams)
    for f, off in zip(fields, vals[1:]):
        assert getattr(dr.DrParams, f).offset == off, f


def test_params_defaults(dr):
    p = dr.dr_params_init()
    assert p.dtype == dr.DR_BF16 and p.x == pytest.approx(1.5) and p.info_scale == 1.0
    assert p.log_floor == pytest.approx(1e-12) and not p.eta and not p.check_finite


def test_status_strings(dr):
    for code in dr.STATUS:
        s = dr.dr_status_string(code)
        assert isinstance(s, str) and s
    assert dr.dr_status_string(12345) == "unknown status"
    # the two-phase GDN/KLA path: one 66560-byte record per (b, h, 64-token chunk)
    assert dr.dr_chunk_fwd_workspace_bytes(1, 1, 8, 2048, 8, 128, 128, 64) == 8 * 8 * 32 * 66560
    assert dr.dr_chunk_fwd_workspace_bytes(0, 1, 2, 65, 3, 128, 128, 64) == 2 * 3 * 2 * 66560
    # PGDN records also carry the write keys and the statistic's chunk map
    assert dr.dr_chunk_fwd_workspace_bytes(2, 1, 4, 4096, 16, 128, 128, 64) == 4 * 16 * 64 * 101376
    # Diagonal KDN: fp32 operand records (either input dtype), then the flags of
    # the variance chain (one per record, a ticket counter and an abort word,
    # rounded up to 256 bytes)
    assert dr.dr_chunk_fwd_workspace_bytes(3, 1, 4, 8192, 16, 128, 128, 64) == \
        4 * 16 * 128 * 135168 + 33024
    assert dr.dr_chunk_fwd_workspace_bytes(3, 0, 1, 65, 1, 128, 128, 64) == 2 * 135168 + 256
    for args in [(1, 0, 8, 2048, 8, 128, 128, 64), (1, 1, 8, 2048, 8, 64, 128, 64),
                 (1, 1, 8, 2048, 8, 128, 128, 32), (3, 1, 8, 2048, 8, 64, 64, 64),
                 (3, 1, 8, 2048, 8, 128, 128, 32)]:
        assert dr.dr_chunk_fwd_workspace_bytes(*args) == 0, args
    assert dr.dr_chunk_fwd_path(dr.DR_KDN, dr.DR_BF16, 128, 128, 64) == "tc_pc_split"
    assert dr.dr_chunk_fwd_path(dr.DR_KDN, dr.DR_FP32, 128, 128, 64) == "simt_split"
    assert dr.dr_chunk_fwd_path(dr.DR_KLA, dr.DR_BF16, 128, 128, 64) == "tc_split"
    assert dr.dr_chunk_fwd_path(dr.DR_PGDN, dr.DR_BF16, 128, 128, 64) == "tc_split"
    assert dr.dr_chunk_fwd_path(dr.DR_KLA, dr.DR_FP32, 64, 64, 64) == "simt"
    # KDA, PKDA and isotropic KDN take Diagonal KDN's two-phase path (same records)
    assert dr.dr_chunk_fwd_path(dr.DR_EKDN, dr.DR_FP32, 64, 64, 16) == "kalman"
    assert dr.dr_chunk_fwd_workspace_bytes(7, 1, 4, 2048, 16, 128, 128, 64) == 0
    for vid in (dr.DR_KDA, dr.DR_PKDA, dr.DR_IKDN):
        assert dr.dr_chunk_fwd_path(vid, dr.DR_BF16, 128, 128, 64) == "tc_pc_split"
        assert dr.dr_chunk_fwd_workspace_bytes(vid, 1, 4, 8192, 16, 128, 128, 64) == \
            dr.dr_chunk_fwd_workspace_bytes(3, 1, 4, 8192, 16, 128, 128, 64)


A = 1 << 20          # a 16-byte aligned address that is never dereferenced
MIS = A + 4          # misaligned


def fwd(dr, variant=1, q=A, k=A, v=A, la=A, out=A, init=None, fin=None, B=1, T=8, H=1, dk=64,
        dv=64, chunk=64, eps=1e-6, **pk):
    p = dr.make_params(**{"dtype": dr.DR_FP32, "eta": A, **pk})
    return dr.dr_chunk_fwd(q, k, v, la, p, variant, eps, init, out, fin, B, T, H, dk, dv, chunk,
                           stream=0)


def test_chunk_fwd_rejects_bad_arguments(dr):
    assert fwd(dr, q=None) == dr.DR_ERR_NULL
    assert fwd(dr, out=None) == dr.DR_ERR_NULL
    assert fwd(dr, eta=None) == dr.DR_ERR_NULL
    assert fwd(dr, variant=2) == dr.DR_ERR_NULL                # PGDN without alphaP/betaP/mu
    assert fwd(dr, variant=3) == dr.DR_ERR_NULL                # KDN without omega/r
    assert fwd(dr, variant=4, eta=None) == dr.DR_ERR_NULL      # KDA without eta
    assert fwd(dr, variant=5) == dr.DR_ERR_NULL                # PKDA without alphaP/betaP/mu
    assert fwd(dr, variant=5, alphaP=A, betaP=A, mu=A, x=0.5) == dr.DR_ERR_ARG
    assert fwd(dr, variant=6, r=A) == dr.DR_ERR_NULL           # isotropic KDN without omega
    assert fwd(dr, variant=7, omega=A) == dr.DR_ERR_NULL       # exact Kalman without r
    assert fwd(dr, variant=8) == dr.DR_ERR_UNSUPPORTED
    assert fwd(dr, dtype=5) == dr.DR_ERR_DTYPE
    assert fwd(dr, dk=96) == dr.DR_ERR_SHAPE
    assert fwd(dr, dv=32) == dr.DR_ERR_SHAPE
    assert fwd(dr, T=0) == dr.DR_ERR_SHAPE
    assert fwd(dr, B=0) == dr.DR_ERR_SHAPE
    assert fwd(dr, chunk=48) == dr.DR_ERR_SHAPE
    assert fwd(dr, eps=-1.0) == dr.DR_ERR_ARG
    assert fwd(dr, variant=2, alphaP=A, betaP=A, mu=A, x=1.0) == dr.DR_ERR_ARG
    assert fwd(dr, variant=3, omega=A, r=A, info_scale=-1.0) == dr.DR_ERR_ARG
    assert fwd(dr, q=MIS) == dr.DR_ERR_ALIGN
    assert fwd(dr, fin=MIS) == dr.DR_ERR_ALIGN
    assert fwd(dr, init=MIS) == dr.DR_ERR_ALIGN
    assert fwd(dr, variant=3, omega=MIS, r=A) == dr.DR_ERR_ALIGN
    assert fwd(dr, variant=7, omega=MIS, r=A) == dr.DR_ERR_ALIGN


def test_decode_rejects_bad_arguments(dr):
    def dec(variant=1, state=A, aux=None, dk=64, **pk):
        p = dr.make_params(**{"dtype": dr.DR_FP32, "eta": A, **pk})
        return dr.dr_decode_step(A, A, A, A, p, variant, 1e-6, state, aux, A, 1, 1, dk, 64,
                                 stream=0)
    assert dec(state=None) == dr.DR_ERR_NULL
    assert dec(variant=2, alphaP=A, betaP=A, mu=A) == dr.DR_ERR_NULL   # aux state required
    assert dec(variant=3, omega=A, r=A) == dr.DR_ERR_NULL
    assert dec(variant=5, alphaP=A, betaP=A, mu=A) == dr.DR_ERR_NULL   # PKDA: aux state required
    assert dec(variant=6, omega=A, r=A) == dr.DR_ERR_NULL              # isotropic KDN: its b
    assert dec(variant=7, omega=A, r=A) == dr.DR_ERR_NULL              # exact Kalman: its P
    assert dec(dk=32) == dr.DR_ERR_SHAPE
    assert dec(state=MIS) == dr.DR_ERR_ALIGN
    assert dec(dtype=2) == dr.DR_ERR_DTYPE


def test_chunk_fwd_workspace_checks(dr):
    """A workspace that is too small or misaligned is refused before any launch."""
    need = dr.dr_chunk_fwd_workspace_bytes(dr.DR_KLA, dr.DR_BF16, 1, 8, 1, 128, 128, 64)
    assert need == 66560
    base = dict(dtype=dr.DR_BF16, dk=128, dv=128)
    assert fwd(dr, workspace=A, workspace_bytes=need - 16, **base) == dr.DR_ERR_WORKSPACE
    assert fwd(dr, workspace=A + 16, workspace_bytes=need, **base) == dr.DR_ERR_ALIGN


def test_backward_refusals_and_workspace_size(dr):
    """dr_chunk_bwd: argument checks before any launch, the supported shapes, and
    the workspace it asks for (the forward's record plus the saved per-chunk data)."""
    A = 1 << 20
    p = dr.make_params(dtype=dr.DR_BF16, eta=A)
    full = dict(dq=A, dk=A, dv=A, d_log_alpha=A, d_eta=A)

    def call(variant=None, B=1, T=64, H=1, d=128, chunk=64, params=None, ws=None, **g):
        pp = params or p
        if ws is not None:
            pp.workspace, pp.workspace_bytes = ws
        grads = dr.make_grads(**{**full, **g})
        return dr.dr_chunk_bwd(A, A, A, A, pp, dr.DR_KLA if variant is None else variant, 1e-6,
                               None, A, None, grads, B, T, H, d, d, chunk, stream=0)

    pg = dr.make_params(dtype=dr.DR_BF16, eta=A, alphaP=A, betaP=A, mu=A)
    assert call(dq=None) == dr.DR_ERR_NULL
    assert call(T=0) == dr.DR_ERR_SHAPE
    assert call(chunk=48) == dr.DR_ERR_SHAPE
    kp = dr.make_params(dtype=dr.DR_BF16, omega=A, r=A)
    assert call(variant=dr.DR_KDN, params=kp) == dr.DR_ERR_NULL        # no d omega, d r
    assert call(variant=dr.DR_KDN, params=kp, d_eta=None, d_omega=A, d_r=A) == dr.DR_ERR_WORKSPACE
    assert call(variant=dr.DR_PKDA, params=dr.make_params(dtype=dr.DR_BF16, eta=A, alphaP=A,
                                                           betaP=A, mu=A)) == dr.DR_ERR_NULL
    assert call(variant=dr.DR_EKDN, params=kp) == dr.DR_ERR_UNSUPPORTED   # no chunkwise form
    assert call(d=64) == dr.DR_ERR_UNSUPPORTED
    assert call(chunk=32) == dr.DR_ERR_UNSUPPORTED
    assert call(params=dr.make_params(dtype=dr.DR_FP32, eta=A)) == dr.DR_ERR_UNSUPPORTED
    assert call(variant=dr.DR_PGDN, params=pg) == dr.DR_ERR_NULL        # no PGDN gate gradients
    assert call() == dr.DR_ERR_WORKSPACE                                # no workspace
    # every array on a 256-byte boundary: the record, S_c, E, dS, E dS^T, dO E^T,
    # dR E^T, gamma <dS, S_c> (PGDN also dL/dw, the key-norm factors, each chunk's part
    # of dL/dmu, each chunk's affine map of the statistic's adjoint and its value at the
    # chunk's end)
    al = lambda x: -(-x // 256) * 256  # noqa: E731
    n, rows = 2 * 3 * 3, 2 * 3
    arrays = [65536, 32768, 65536, 32768, 16384, 16384]
    need = dr.dr_chunk_bwd_workspace_bytes(dr.DR_KLA, dr.DR_BF16, 2, 130, 3, 128, 128, 64)
    assert need == al(n * 66560) + sum(al(n * x) for x in arrays) + al(4 * n)
    need_p = dr.dr_chunk_bwd_workspace_bytes(dr.DR_PGDN, dr.DR_BF16, 2, 130, 3, 128, 128, 64)
    assert need_p == (al(n * 101376) + sum(al(n * x) for x in arrays) + al(4 * n) + al(n * 32768)
                      + al(n * 256) + al(4 * n) + al(n * 1024) + al(n * 512))
    # per-channel decay (KDA): the per-channel record and the forward's hand-over
    # flags, gamma_c <dS_c, S_c> per channel, the forward's write vectors
    chain = -(-((n + 2) * 4) // 256) * 256
    need_a = dr.dr_chunk_bwd_workspace_bytes(dr.DR_KDA, dr.DR_BF16, 2, 130, 3, 128, 128, 64)
    assert need_a == (al(n * 135168 + chain) + sum(al(n * x) for x in arrays) + al(4 * 128 * n)
                      + al(n * 32768))
    assert call(ws=(A, 1000)) == dr.DR_ERR_WORKSPACE
    assert call(ws=(A + 16, 1 << 30)) == dr.DR_ERR_ALIGN
    # Diagonal KDN, PKDA, isotropic KDN: as KDA plus dL/dw, 4 B per chunk, each
    # chunk's affine map of the gain adjoint and the adjoint at its end
    need_k = dr.dr_chunk_bwd_workspace_bytes(dr.DR_KDN, dr.DR_BF16, 2, 130, 3, 128, 128, 64)
    assert need_k == need_a + al(n * 32768) + al(4 * n) + al(n * 1024) + al(n * 512)
    for vid in (dr.DR_PKDA, dr.DR_IKDN):   # the same layout (with PKDA's chunks' dL/dmu parts)
        assert dr.dr_chunk_bwd_workspace_bytes(vid, dr.DR_BF16, 2, 130, 3, 128, 128, 64) == need_k
    assert dr.dr_chunk_bwd_workspace_bytes(dr.DR_EKDN, dr.DR_BF16, 1, 64, 1, 128, 128, 64) == 0


def test_grads_struct_layout_matches_c(dr):
    fields = [f for f, _ in dr.DrGrads._fields_]
    src = "#include <stdio.h>\n#include <stddef.h>\n#include \"dr.h\"\nint main(void){\n"
    src += 'printf("%zu\\n", sizeof(dr_grads));\n'
    for f in fields:
        src += f'printf("%zu\\n", offsetof(dr_grads, {f}));\n'
    src += "return 0;}\n"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "g.c")
        exe = os.path.join(d, "g")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        out = [int(x) for x in subprocess.run([exe], capture_output=True, text=True,
                                              check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(dr.DrGrads)
    assert out[1:] == [getattr(dr.DrGrads, f).offset for f in fields]
