"""dr_chunk_fwd_noalloc: the two-phase forward on the library's own scratch.

Some callers cannot allocate device memory (a framework whose allocator owns
all of it, a real-time loop that cannot take cudaMalloc's synchronisation, a
plug-in given only its input and output buffers), so they cannot supply the
workspace dr_chunk_fwd wants for its fastest path.  This entry point keeps the
per-chunk records in a fixed library-owned device array instead.

The GPU test calls it through the C ABI twice in a row, on different inputs, so
the second call runs over the first call's leftover records, and compares each
result with dr_chunk_fwd on a caller-allocated workspace: the same kernels on the
same inputs, so the same bits.  The host test covers the refusals that happen before any CUDA call.
This file is collected last on purpose.
"""

import pytest
import torch

from recurrent_associative_memory_gb300 import workloads as W

A = 1 << 20   # a 16-byte aligned address that is never dereferenced (refused calls only)


def test_noalloc_refusals_on_host():
    from recurrent_associative_memory_gb300 import dr

    def call(B=1, T=64, H=1, dk=128, dv=128, chunk=64, dtype=None, variant=None):
        p = dr.make_params(dtype=dr.DR_BF16 if dtype is None else dtype, eta=A)
        return dr.dr_chunk_fwd_noalloc(A, A, A, A, p, dr.DR_KLA if variant is None else variant,
                                       1e-6, None, A, None, B, T, H, dk, dv, chunk, stream=0)

    max_records = dr.DR_NOALLOC_SCRATCH_BYTES // 66560
    assert max_records == 1008
    assert call(T=64 * (max_records + 1)) == dr.DR_ERR_WORKSPACE
    assert call(B=2, T=64 * 64, H=8) == dr.DR_ERR_WORKSPACE          # 2*8*64 = 1024 records
    assert call(dk=64) == dr.DR_ERR_UNSUPPORTED
    assert call(chunk=32) == dr.DR_ERR_UNSUPPORTED
    assert call(dtype=dr.DR_FP32) == dr.DR_ERR_UNSUPPORTED
    assert call(variant=dr.DR_KDN, dk=64, dv=64) == dr.DR_ERR_UNSUPPORTED
    assert call(T=0) == dr.DR_ERR_SHAPE
    # the per-channel-decay records (135,168 bytes) and the chain flags after them
    p = dr.make_params(dtype=dr.DR_FP32, omega=A, r=A)
    kcall = lambda T: dr.dr_chunk_fwd_noalloc(A, A, A, A, p, dr.DR_KDN, 1e-6, None, A, None,  # noqa: E731
                                              1, T, 1, 128, 128, 64, stream=0)
    assert kcall(64 * 497) == dr.DR_ERR_WORKSPACE                        # 497 records
    assert dr.dr_chunk_fwd_workspace_bytes(dr.DR_KDN, dr.DR_FP32, 1, 64 * 496, 1, 128, 128, 64) \
        <= dr.DR_NOALLOC_SCRATCH_BYTES
    # the same answers as dr_chunk_fwd for a bad dtype or a missing pointer
    assert call(dtype=7) == dr.DR_ERR_DTYPE
    bad = dr.make_params(dtype=dr.DR_BF16, eta=A)
    assert dr.dr_chunk_fwd_noalloc(A, None, A, A, bad, dr.DR_KLA, 1e-6, None, A, None,
                                   1, 64, 1, 128, 128, 64, stream=0) == dr.DR_ERR_NULL
    assert dr.dr_chunk_fwd(A, None, A, A, bad, dr.DR_KLA, 1e-6, None, A, None,
                           1, 64, 1, 128, 128, 64, stream=0) == dr.DR_ERR_NULL


@pytest.mark.gpu
def test_noalloc_matches_chunk_fwd_on_two_calls():
    from recurrent_associative_memory_gb300 import dr, runner

    cases = [("kla", 2, 333, 3, 31), ("gdn", 1, 64 * 40 + 9, 8, 32)]   # 36 then 328 records
    g = torch.Generator().manual_seed(30)
    for variant, B, T, H, seed in cases:
        wl = W.small("gdn_kla_bf16", B=B, T=T, H=H, seed=seed)
        dev = runner.to_device(W.generate(wl, variant))
        S0 = (0.3 * torch.randn(B, H, 128, 128, generator=g)).cuda()
        ref_out, ref_S, _ = runner.chunk_fwd(dev, init_state=S0)   # dr_chunk_fwd + own workspace
        out = torch.empty_like(ref_out)
        S = torch.empty_like(ref_S)
        st = dr.dr_chunk_fwd_noalloc(dev["q"], dev["k"], dev["v"], dev["log_alpha"],
                                     runner.params_for(dev), dr.VARIANT_IDS[variant],
                                     dev.get("eps", 1e-6), S0, out, S, B, T, H, 128, 128, 64)
        dr.check(st, "dr_chunk_fwd_noalloc")
        torch.cuda.synchronize()
        assert dr.dr_get_device_status() == 0
        # the same kernels on the same inputs: the same bits
        assert torch.equal(out, ref_out) and torch.equal(S, ref_S), variant


@pytest.mark.gpu
def test_noalloc_per_channel_decay_paths_match_chunk_fwd():
    """The library-owned scratch serves the CUDA-core two-phase path too: Diagonal
    KDN with its variance chain (many rows: the chain's flags live after the
    records in the scratch), KDA, and isotropic KDN; same bits as a caller
    workspace."""
    from recurrent_associative_memory_gb300 import dr, runner

    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    Hc = max(26, -(-nsm // 6))          # 3 B H >= SM count: the chained prep runs
    cases = [("kdn", "kdn_bf16", 2, 100, Hc), ("kda", "kda_bf16", 2, 130, 3),
             ("ikdn", "ikdn_bf16", 2, 77, Hc)]
    for variant, base, B, T, H in cases:
        if variant != "kda":
            assert 3 * B * H >= nsm and B * H * ((T + 63) // 64) <= 496
        wl = W.small(base, B=B, T=T, H=H, seed=40)
        dev = runner.to_device(W.generate(wl, variant))
        ref_out, ref_S, ref_aux = runner.chunk_fwd(dev)
        out, S = torch.empty_like(ref_out), torch.empty_like(ref_S)
        aux = None if ref_aux is None else torch.empty_like(ref_aux)
        p = runner.params_for(dev, aux_final=aux)
        st = dr.dr_chunk_fwd_noalloc(dev["q"], dev["k"], dev["v"], dev["log_alpha"], p,
                                     dr.VARIANT_IDS[variant], dev.get("eps", 1e-6), None, out, S,
                                     B, T, H, 128, 128, 64)
        dr.check(st, "dr_chunk_fwd_noalloc")
        torch.cuda.synchronize()
        assert dr.dr_get_device_status() == 0
        assert torch.equal(out, ref_out) and torch.equal(S, ref_S), variant
        if aux is not None:
            assert torch.equal(aux, ref_aux), variant
