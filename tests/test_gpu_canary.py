"""Canary guard bytes around every buffer the library writes (the stand-in for a memory checker).

Every entry point is called through the C ABI with each output, workspace and debug-dump buffer
placed inside a larger allocation whose 4 KiB before and after are filled with a fixed pattern.
After the call and a device synchronisation the guards must hold the pattern, and the inputs must
be unchanged.  Shapes with a ragged last key tile (N = 320), causal masking, Q-smoothing and both
head dimensions exercise every edge of the kernels' index arithmetic.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """``nbytes`` of device memory (256-byte aligned) between two guard regions."""

    def __init__(self, nbytes: int, fill: int | None = None):
        self.n = int(nbytes)
        self.buf = torch.full((GUARD + self.n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        if fill is not None:
            self.buf[GUARD:GUARD + self.n] = fill

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + GUARD

    def view(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.n].view(dtype).view(shape)

    def intact(self) -> bool:
        b = self.buf
        return bool((b[:GUARD] == PATTERN).all() and (b[GUARD + self.n:] == PATTERN).all())


def _lib():
    from bit_trainable_attention_sage_gb300 import build
    build.build()
    import bit_trainable_attention_sage_gb300 as sg
    return sg, sg.lib()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _inputs(B, H, N, d, dt, seed):
    g = torch.Generator().manual_seed(seed)
    t = [torch.randn((B, H, N, d), generator=g).to(dt).cuda() for _ in range(4)]
    t[3] = t[3] * 0.1
    return t


def _check(bufs, inputs, snapshots, what):
    torch.cuda.synchronize()
    for name, b in bufs.items():
        assert b.intact(), (what, name, "guard bytes overwritten")
    for t, s in zip(inputs, snapshots):
        assert torch.equal(t, s), (what, "an input was modified")


CASES = [
    (1, 2, 320, 128, torch.float16, True, False),
    (2, 1, 320, 64, torch.bfloat16, False, True),
    (1, 3, 192, 64, torch.float16, True, True),
]


@pytest.mark.parametrize("B,H,N,d,dt,causal,smooth_q", CASES)
def test_sagebwd_calls_stay_inside_their_buffers(B, H, N, d, dt, causal, smooth_q):
    sg, L = _lib()
    code = 0 if dt == torch.float16 else 1
    n, rows, nb = B * H * N * d, B * H * N, B * H * (N // 64)
    Q, K, V, dO = _inputs(B, H, N, d, dt, seed=N + d)
    snaps = [t.clone() for t in (Q, K, V, dO)]
    es = 2
    for dump, ops in ((False, False), (True, False), (False, True)):
        bufs = {}
        p = sg.make_params(B, H, N, d, code, causal, smooth_q=smooth_q)
        if ops:
            # SAGE_FLAG_OPS16: the quantiser also writes the codes' fp16 values, which the
            # forward and backward then read
            bufs["ops16"] = Guarded(3 * 2 * n)
            p.flags |= sg.binding.SAGE_FLAG_OPS16
            p.ops16 = bufs["ops16"].ptr
        # ---- quantise (with workspace), then the allocation-free variant into fresh buffers
        for k, nbytes in (("Qh", n), ("Kh", n), ("Vh", n), ("sQ", 4 * nb), ("sK", 4 * nb), ("sV", 4 * nb),
                          ("muK", 4 * B * H * d), ("muQ", 4 * nb * d)):
            bufs[k] = Guarded(nbytes)
        wq = L.sage_quantize_workspace_bytes(ctypes.byref(p))
        bufs["ws_q"] = Guarded(max(wq, 16))
        st = L.sage_quantize_smooth(ctypes.byref(p), Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                                    *[bufs[k].ptr for k in ("Qh", "Kh", "Vh", "sQ", "sK", "sV", "muK", "muQ")],
                                    bufs["ws_q"].ptr, wq, _stream())
        assert st == 0
        _check(bufs, (Q, K, V), snaps[:3], "sage_quantize_smooth")
        na = {k: Guarded(bufs[k].n) for k in ("Qh", "Kh", "Vh", "sQ", "sK", "sV", "muK", "muQ")}
        pn = sg.make_params(B, H, N, d, code, causal, smooth_q=smooth_q)
        if ops:
            na["ops16"] = Guarded(3 * 2 * n)
            pn.flags |= sg.binding.SAGE_FLAG_OPS16
            pn.ops16 = na["ops16"].ptr
        st = L.sage_quantize_smooth_noalloc(ctypes.byref(pn), Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                                            *[na[k].ptr for k in ("Qh", "Kh", "Vh", "sQ", "sK", "sV", "muK", "muQ")],
                                            _stream())
        assert st == 0
        _check(na, (Q, K, V), snaps[:3], "sage_quantize_smooth_noalloc")
        # ---- forward (optionally with the debug dump)
        pf = sg.make_params(B, H, N, d, code, causal, smooth_q=smooth_q)
        if ops:
            pf.flags |= sg.binding.SAGE_FLAG_OPS16
            pf.ops16 = bufs["ops16"].ptr
        if dump:
            bufs["dump_f"] = Guarded(L.sage_dump_bytes(ctypes.byref(pf), 0))
            pf.flags |= sg.binding.SAGE_FLAG_DUMP
            pf.dump = bufs["dump_f"].ptr
            pf.dump_bytes = bufs["dump_f"].n
        bufs["O"] = Guarded(es * n)
        bufs["L"] = Guarded(4 * rows)
        wf = L.sage_fwd_workspace_bytes(ctypes.byref(pf))
        bufs["ws_f"] = Guarded(wf)
        qp = [bufs[k].ptr for k in ("Qh", "Kh", "Vh", "sQ", "sK", "sV")]
        st = L.sage_attn_fwd(ctypes.byref(pf), *qp, K.data_ptr() if smooth_q else None,
                             bufs["muK"].ptr if smooth_q else None, bufs["muQ"].ptr if smooth_q else None,
                             bufs["O"].ptr, bufs["L"].ptr, bufs["ws_f"].ptr, wf, _stream())
        assert st == 0
        _check(bufs, (Q, K, V), snaps[:3], f"sage_attn_fwd dump={dump} ops16={ops}")
        # ---- backward (optionally with the debug dump)
        pb = sg.make_params(B, H, N, d, code, causal, smooth_q=smooth_q)
        if ops:
            pb.flags |= sg.binding.SAGE_FLAG_OPS16
            pb.ops16 = bufs["ops16"].ptr
        if dump:
            bufs["dump_b"] = Guarded(L.sage_dump_bytes(ctypes.byref(pb), 1))
            pb.flags |= sg.binding.SAGE_FLAG_DUMP
            pb.dump = bufs["dump_b"].ptr
            pb.dump_bytes = bufs["dump_b"].n
        for k in ("dQ", "dK", "dV"):
            bufs[k] = Guarded(4 * n)
        wb = L.sage_bwd_workspace_bytes(ctypes.byref(pb))
        bufs["ws_b"] = Guarded(wb)
        st = L.sage_attn_bwd(ctypes.byref(pb), bufs["Qh"].ptr, bufs["Kh"].ptr, bufs["sQ"].ptr, bufs["sK"].ptr,
                             K.data_ptr() if smooth_q else None, bufs["muK"].ptr if smooth_q else None,
                             bufs["muQ"].ptr if smooth_q else None, V.data_ptr(), bufs["O"].ptr, bufs["L"].ptr,
                             dO.data_ptr(), bufs["dQ"].ptr, bufs["dK"].ptr, bufs["dV"].ptr, bufs["ws_b"].ptr, wb,
                             _stream())
        assert st == 0
        _check(bufs, (Q, K, V, dO), snaps, f"sage_attn_bwd dump={dump} ops16={ops}")
        assert sg.sage_device_status() == 0


@pytest.mark.parametrize("B,H,N,d,dt,causal,smooth_q", CASES[:2])
def test_variant_calls_stay_inside_their_buffers(B, H, N, d, dt, causal, smooth_q):
    """QK-norm, its gradient, the FP4 forward and the three Attn-QAT calls."""
    sg, L = _lib()
    code = 0 if dt == torch.float16 else 1
    n, rows, nb = B * H * N * d, B * H * N, B * H * (N // 64)
    Q, K, V, dO = _inputs(B, H, N, d, dt, seed=7 * N + d)
    snaps = [t.clone() for t in (Q, K, V, dO)]
    es = 2
    # ---- QK-norm prologue (with normalised outputs) and its gradient
    p = sg.make_params(B, H, N, d, code, causal, smooth_q=smooth_q)
    bufs = {k: Guarded(nbytes) for k, nbytes in (
        ("Qh", n), ("Kh", n), ("Vh", n), ("sQ", 4 * nb), ("sK", 4 * nb), ("sV", 4 * nb), ("muK", 4 * B * H * d),
        ("muQ", 4 * nb * d), ("rQ", 4 * rows), ("rK", 4 * rows), ("Qn", es * n), ("Kn", es * n))}
    gam = Guarded(4 * d, fill=0)
    gam.view(torch.float32, (d,)).fill_(1.25)
    wq = L.sage_quantize_workspace_bytes(ctypes.byref(p))
    bufs["ws_q"] = Guarded(max(wq, 16))
    qn = sg.binding.SageQkNorm(gam.ptr, gam.ptr, 1e-6, bufs["rQ"].ptr, bufs["rK"].ptr, bufs["Qn"].ptr, bufs["Kn"].ptr)
    st = L.sage_quantize_smooth_qknorm(ctypes.byref(p), ctypes.byref(qn), Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                                       *[bufs[k].ptr for k in ("Qh", "Kh", "Vh", "sQ", "sK", "sV", "muK", "muQ")],
                                       bufs["ws_q"].ptr, wq, _stream())
    assert st == 0
    _check(bufs, (Q, K, V), snaps[:3], "sage_quantize_smooth_qknorm")
    dY = torch.randn((B, H, N, d), device="cuda")
    bufs["dX"] = Guarded(4 * n)
    bufs["dg"] = Guarded(4 * d)
    st = L.sage_qknorm_bwd(ctypes.byref(p), Q.data_ptr(), gam.ptr, bufs["rQ"].ptr, dY.data_ptr(),
                           bufs["dX"].ptr, bufs["dg"].ptr, _stream())
    assert st == 0
    _check(bufs, (Q, K, V), snaps[:3], "sage_qknorm_bwd")
    # ---- FP4 inference forward
    p4 = sg.make_params(B, H, N, d, code, causal, smooth_q=smooth_q)
    f4 = {k: Guarded(nbytes) for k, nbytes in (
        ("Qc", n // 2), ("Kc", n // 2), ("Vc", n // 2), ("sQ", n // 16), ("sK", n // 16), ("sV", n // 16),
        ("muK", 4 * B * H * d), ("muQ", 4 * nb * d), ("O", es * n), ("L", 4 * rows))}
    f4["ws_q"] = Guarded(max(wq, 16))
    st = L.sage_quantize_fp4(ctypes.byref(p4), Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                             *[f4[k].ptr for k in ("Qc", "Kc", "Vc", "sQ", "sK", "sV", "muK", "muQ")],
                             f4["ws_q"].ptr, wq, _stream())
    assert st == 0
    wf = L.sage_fwd_workspace_bytes(ctypes.byref(p4))
    f4["ws_f"] = Guarded(wf)
    st = L.sage_attn_fwd_fp4(ctypes.byref(p4), *[f4[k].ptr for k in ("Qc", "Kc", "Vc", "sQ", "sK", "sV")],
                             K.data_ptr() if smooth_q else None, f4["muK"].ptr if smooth_q else None,
                             f4["muQ"].ptr if smooth_q else None, f4["O"].ptr, f4["L"].ptr, f4["ws_f"].ptr, wf,
                             _stream())
    assert st == 0
    _check(f4, (Q, K, V), snaps[:3], "FP4 quantise + forward")
    # ---- Attn-QAT
    pq = sg.make_params(B, H, N, d, code, causal, smooth_k=False)
    qa = {k: Guarded(nbytes) for k, nbytes in (
        ("Qf", es * n), ("Kf", es * n), ("Vf", es * n), ("O", es * n), ("Op", 4 * n), ("L", 4 * rows),
        ("R", 4 * nb * N), ("dQ", 4 * n), ("dK", 4 * n), ("dV", 4 * n))}
    st = L.sage_qat_quantize(ctypes.byref(pq), Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                             qa["Qf"].ptr, qa["Kf"].ptr, qa["Vf"].ptr, _stream())
    assert st == 0
    st = L.sage_qat_fwd(ctypes.byref(pq), qa["Qf"].ptr, qa["Kf"].ptr, qa["Vf"].ptr, qa["O"].ptr, qa["Op"].ptr,
                        qa["L"].ptr, qa["R"].ptr, _stream())
    assert st == 0
    wb = L.sage_qat_bwd_workspace_bytes(ctypes.byref(pq))
    qa["ws_b"] = Guarded(wb)
    st = L.sage_qat_bwd(ctypes.byref(pq), qa["Qf"].ptr, qa["Kf"].ptr, qa["Vf"].ptr, qa["Op"].ptr, qa["L"].ptr,
                        qa["R"].ptr, dO.data_ptr(), qa["dQ"].ptr, qa["dK"].ptr, qa["dV"].ptr, qa["ws_b"].ptr, wb,
                        _stream())
    assert st == 0
    _check(qa, (Q, K, V, dO), snaps, "Attn-QAT quantise + forward + backward")
    assert sg.sage_device_status() == 0
    assert np.isfinite(qa["dQ"].view(torch.float32, (n,)).cpu().numpy()).all()
