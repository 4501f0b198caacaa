"""The C-ABI library: it loads, exports every entry point include/sage.h declares, sizes its
workspaces, and rejects bad arguments before touching the GPU (CPU-only checks)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sg():
    from bit_trainable_attention_sage_gb300 import build
    build.build()
    import bit_trainable_attention_sage_gb300 as sg
    return sg


def _declared():
    text = open(os.path.join(ROOT, "include", "sage.h")).read()
    return sorted(set(re.findall(r"SAGE_API\s+[\w\s\*]+?\b(sage_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("sage_quantize_smooth", "sage_attn_fwd", "sage_attn_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(sg):
    L = sg.lib()
    for name in _declared():
        assert hasattr(L, name), name
    assert "sm_103a" in sg.sage_version()


def test_workspace_sizes(sg):
    L = sg.lib()
    p = sg.make_params(2, 16, 8192, 128, 0, False)
    n = 2 * 16 * 8192 * 128
    fwd = L.sage_fwd_workspace_bytes(ctypes.byref(p))
    bwd = L.sage_bwd_workspace_bytes(ctypes.byref(p))
    assert fwd >= 3 * 2 * n
    assert bwd >= 3 * 2 * n + 4 * 2 * 16 * 8192
    pq = sg.make_params(2, 16, 8192, 128, 0, False, smooth_q=True)
    assert L.sage_fwd_workspace_bytes(ctypes.byref(pq)) >= fwd + 4 * 2 * 16 * 128 * 8192
    bad = sg.make_params(1, 1, 100, 128, 0, False)
    assert L.sage_fwd_workspace_bytes(ctypes.byref(bad)) == 0
    # the INT8-dP ablation adds the V codes (1 B), their fp16 copy (2 B) and the block scales
    p8 = sg.make_params(2, 16, 8192, 128, 0, False)
    p8.flags = sg.binding.SAGE_FLAG_DP_INT8
    extra = L.sage_bwd_workspace_bytes(ctypes.byref(p8)) - bwd
    assert 3 * n + 4 * 2 * 16 * 128 <= extra <= 3 * n + 4 * 2 * 16 * 128 + 3 * 256


def test_fp8_flag_checks(sg):
    """SAGE_FLAG_FP8 is accepted alone (same workspaces as INT8) and refused with the dump or with
    INT8 dP (SAGE_ERR_UNSUPPORTED) before any launch."""
    L = sg.lib()
    p = sg.make_params(1, 2, 256, 128, 0, False)
    pf = sg.make_params(1, 2, 256, 128, 0, False, fp8=True)
    assert pf.flags == sg.binding.SAGE_FLAG_FP8
    for q in ("sage_quantize_workspace_bytes", "sage_fwd_workspace_bytes", "sage_bwd_workspace_bytes"):
        assert getattr(L, q)(ctypes.byref(pf)) == getattr(L, q)(ctypes.byref(p)) > 0 or q == "sage_quantize_workspace_bytes"
    for extra in (sg.binding.SAGE_FLAG_DUMP, sg.binding.SAGE_FLAG_DP_INT8):
        bad = sg.make_params(1, 2, 256, 128, 0, False, fp8=True)
        bad.flags |= extra
        assert L.sage_attn_fwd(ctypes.byref(bad), *[_fake(i) for i in range(12)], 1 << 30, None) == 2
        assert L.sage_attn_bwd(ctypes.byref(bad), *[_fake(i) for i in range(15)], 1 << 30, None) == 2


def _fake(i):
    return 0x10000 * (i + 1)    # aligned non-null addresses; never dereferenced (calls fail first)


@pytest.mark.parametrize("field,value,status", [
    ("d", 96, 2), ("N", 100, 2), ("dtype", 7, 2), ("B", 0, 1), ("causal", 2, 1), ("flags", 8, 1),
])
def test_bad_params_rejected(sg, field, value, status):
    L = sg.lib()
    p = sg.make_params(1, 1, 128, 64, 0, False)
    setattr(p, field, value)
    args = [_fake(i) for i in range(12)]
    st = L.sage_attn_fwd(ctypes.byref(p), *args, 1 << 30, None)
    assert st == status
    assert sg.sage_status_string(st)


def test_null_misaligned_and_workspace(sg):
    L = sg.lib()
    p = sg.make_params(1, 1, 128, 64, 0, False)
    args = [_fake(i) for i in range(12)]
    args[0] = None
    assert L.sage_attn_fwd(ctypes.byref(p), *args, 1 << 30, None) == 1
    args = [_fake(i) for i in range(12)]
    args[3] = _fake(3) + 4
    assert L.sage_attn_fwd(ctypes.byref(p), *args, 1 << 30, None) == 3
    args = [_fake(i) for i in range(12)]
    assert L.sage_attn_fwd(ctypes.byref(p), *args, 16, None) == 6
    args = [_fake(i) for i in range(15)]
    assert L.sage_attn_bwd(ctypes.byref(p), *args, 16, None) == 6
    qargs = [_fake(i) for i in range(12)]
    qargs[9] = None   # muK
    assert L.sage_quantize_smooth(ctypes.byref(p), *qargs, 1 << 30, None) == 1


def test_ops16_flag_checks(sg):
    """SAGE_FLAG_OPS16 needs a 16-byte aligned p->ops16 (SAGE_ERR_ARG / SAGE_ERR_ALIGN), drops the
    widened operand copies from the forward (3 of them) and backward (2) workspaces, and is refused
    by the FP4 entry points (fake device pointers are never dereferenced)."""
    L = sg.lib()
    n = 1 * 2 * 256 * 128
    p = sg.make_params(1, 2, 256, 128, 0, False)
    po = sg.make_params(1, 2, 256, 128, 0, False)
    po.flags |= sg.binding.SAGE_FLAG_OPS16
    po.ops16 = _fake(30)
    # the copies sit first in both workspaces, each 256-byte aligned
    assert L.sage_fwd_workspace_bytes(ctypes.byref(p)) - L.sage_fwd_workspace_bytes(ctypes.byref(po)) == 3 * 2 * n
    assert L.sage_bwd_workspace_bytes(ctypes.byref(p)) - L.sage_bwd_workspace_bytes(ctypes.byref(po)) == 2 * 2 * n
    assert L.sage_quantize_workspace_bytes(ctypes.byref(po)) == L.sage_quantize_workspace_bytes(ctypes.byref(p))
    args = [_fake(i) for i in range(12)]
    po.ops16 = None
    assert L.sage_attn_fwd(ctypes.byref(po), *args, 1 << 30, None) == 1
    po.ops16 = _fake(30) + 8
    assert L.sage_attn_fwd(ctypes.byref(po), *args, 1 << 30, None) == 3
    assert L.sage_quantize_smooth(ctypes.byref(po), *args, 1 << 30, None) == 3
    po.ops16 = _fake(30)
    assert L.sage_quantize_fp4(ctypes.byref(po), *args, 1 << 30, None) == 2
    assert L.sage_attn_fwd_fp4(ctypes.byref(po), *args, 1 << 30, None) == 2


def test_qknorm_argument_checks(sg):
    """The QK-norm calls refuse bad arguments before any launch (fake device pointers are never
    dereferenced)."""
    L = sg.lib()
    p = sg.make_params(1, 1, 128, 64, 0, False)
    args = [_fake(i) for i in range(12)]
    QN = sg.binding.SageQkNorm

    def call(qn, params=p):
        return L.sage_quantize_smooth_qknorm(ctypes.byref(params), None if qn is None else ctypes.byref(qn),
                                             *args, 1 << 30, None)

    assert call(None) == 1
    assert call(QN(None, None, -1.0, _fake(20), _fake(21), None, None)) == 1
    assert call(QN(None, None, float("nan"), _fake(20), _fake(21), None, None)) == 1
    assert call(QN(None, None, float("inf"), _fake(20), _fake(21), None, None)) == 1
    assert call(QN(None, None, 1e-6, None, _fake(21), None, None)) == 1
    assert call(QN(None, None, 1e-6, _fake(20) + 4, _fake(21), None, None)) == 3
    assert call(QN(_fake(22) + 8, None, 1e-6, _fake(20), _fake(21), None, None)) == 3
    psq = sg.make_params(1, 1, 128, 64, 0, False, smooth_q=True)
    assert call(QN(None, None, 1e-6, _fake(20), _fake(21), None, None), psq) == 1    # smooth_q needs Kn
    bad = sg.make_params(1, 1, 100, 64, 0, False)
    assert call(QN(None, None, 1e-6, _fake(20), _fake(21), None, None), bad) == 2
    # the gradient call: null input, dX aliasing dY, misaligned gamma
    f = [_fake(i) for i in range(6)]
    assert L.sage_qknorm_bwd(ctypes.byref(p), None, None, f[2], f[3], f[4], None, None) == 1
    assert L.sage_qknorm_bwd(ctypes.byref(p), f[1], None, f[2], f[3], f[3], None, None) == 1
    assert L.sage_qknorm_bwd(ctypes.byref(p), f[1], f[0] + 4, f[2], f[3], f[4], None, None) == 3


def test_qat_argument_checks(sg):
    """The Attn-QAT calls take no flags and no smoothing (SAGE_ERR_UNSUPPORTED), refuse null and
    misaligned pointers and a short workspace, all before any launch (fake device pointers are
    never dereferenced).  Their workspace holds D and L2: two 256-byte-aligned float rows."""
    L = sg.lib()
    p = sg.make_params(1, 2, 128, 64, 0, False, smooth_k=False)
    f = [_fake(i) for i in range(12)]
    assert L.sage_qat_bwd_workspace_bytes(ctypes.byref(p)) == 2 * 1024
    for bad in (sg.make_params(1, 2, 128, 64, 0, False), sg.make_params(1, 2, 128, 64, 0, False, smooth_k=False, smooth_q=True),
                sg.make_params(1, 2, 128, 64, 0, False, smooth_k=False, fp8=True)):
        assert L.sage_qat_quantize(ctypes.byref(bad), *f[:6], None) == 2
        assert L.sage_qat_fwd(ctypes.byref(bad), *f[:7], None) == 2
        assert L.sage_qat_bwd(ctypes.byref(bad), *f[:10], f[11], 1 << 20, None) == 2
        assert L.sage_qat_bwd_workspace_bytes(ctypes.byref(bad)) == 0
    assert L.sage_qat_quantize(ctypes.byref(p), f[0], None, *f[2:6], None) == 1
    assert L.sage_qat_fwd(ctypes.byref(p), *f[:6], f[6] + 4, None) == 3
    assert L.sage_qat_bwd(ctypes.byref(p), *f[:10], f[11], 100, None) == 6
    assert L.sage_qat_bwd(ctypes.byref(p), *f[:10], None, 1 << 20, None) == 6
    assert L.sage_qat_bwd(ctypes.byref(p), *f[:9], f[9] + 8, f[11], 1 << 20, None) == 3


def test_noalloc_partials_query(sg):
    """The allocation-free quantise call needs (456 + B*H)*d + B*H float64 words of K-mean scratch
    with K-smoothing (a partial-sum slot of d for each of the pass's at most 456 CTAs and each
    head, and a word of two 32-bit counters for each head) and none without; the host-only query
    says so, and returns 0 for parameters the call would refuse."""
    L = sg.lib()
    cap = L.sage_quantize_noalloc_max_partials()
    assert cap == 131072
    for B, H, N, d in ((1, 3, 320, 64), (2, 16, 8192, 128), (1, 563, 8192, 128), (1, 564, 8192, 128)):
        p = sg.make_params(B, H, N, d, 0, False)
        assert L.sage_quantize_noalloc_partials_needed(ctypes.byref(p)) == (456 + B * H) * d + B * H
    # at d = 128, B*H = 564 exceeds the array and 563 fits
    assert L.sage_quantize_noalloc_partials_needed(ctypes.byref(sg.make_params(1, 564, 8192, 128, 0, False))) > cap
    assert L.sage_quantize_noalloc_partials_needed(ctypes.byref(sg.make_params(1, 563, 8192, 128, 0, False))) <= cap
    assert L.sage_quantize_noalloc_partials_needed(ctypes.byref(sg.make_params(1, 2, 256, 64, 0, False, smooth_k=False))) == 0
    assert L.sage_quantize_noalloc_partials_needed(ctypes.byref(sg.make_params(1, 2, 100, 64, 0, False))) == 0


def test_binding_types_every_declared_call(sg):
    """Every entry point the header declares gets its argument types when the binding loads the
    library: a ctypes call without them passes 64-bit pointers as C ints."""
    L = sg.lib()
    for name in _declared():
        assert getattr(L, name).argtypes is not None, name
