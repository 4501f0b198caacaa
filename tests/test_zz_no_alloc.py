"""sage_quantize_smooth_noalloc: the quantise step for callers that cannot allocate device memory
while they run (for example a plug-in whose host framework owns all device memory, or a loop that
must not wait on an allocation).  It keeps its K-mean scratch in a fixed array inside the library.

Checked through the C ABI against sage_quantize_smooth, two calls in a row on different inputs
(the second call reuses the array the first one left behind): codes, scales and means must be
bit-identical, the same bar the other quantise tests use.  Also: a problem larger than the array
is refused with SAGE_ERR_WORKSPACE before anything is launched.

This file is collected last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _inputs(B, H, N, d, dtype, seed, offset):
    g = torch.Generator().manual_seed(seed)
    shape = (B, H, N, d)
    Q, K, V = (torch.randn(shape, generator=g) for _ in range(3))
    K = K + offset * torch.randn((1, H, 1, d), generator=g)     # a shared K offset to smooth away
    return [t.to(dtype).cuda().contiguous() for t in (Q, K, V)]


def _same(a, b):
    if a is None or b is None:
        return a is None and b is None
    return torch.equal(a.view(torch.int8) if a.dtype != torch.int8 else a,
                       b.view(torch.int8) if b.dtype != torch.int8 else b)


@pytest.mark.parametrize("B,H,N,d,dtype,smooth_q", [
    (2, 4, 512, 128, torch.float16, False),
    (1, 3, 320, 64, torch.bfloat16, True),
])
def test_noalloc_matches_quantize_two_calls(B, H, N, d, dtype, smooth_q):
    from bit_trainable_attention_sage_gb300 import build
    build.build()
    import bit_trainable_attention_sage_gb300 as sg
    for call, (seed, offset) in enumerate(((1, 3.0), (2, -5.0))):
        Q, K, V = _inputs(B, H, N, d, dtype, seed, offset)
        ref = sg.sage_quantize_smooth(Q, K, V, smooth_q=smooth_q)
        got = sg.sage_quantize_smooth_noalloc(Q, K, V, smooth_q=smooth_q)
        assert sg.sage_device_status() == 0
        for name in ("Qh", "Kh", "Vh", "sQ", "sK", "sV", "muK", "muQ"):
            assert _same(getattr(got, name), getattr(ref, name)), (call, name)


def test_noalloc_rejects_beyond_capacity():
    """B*H = 2048 heads of d = 128 need (456 + 2048) * 128 partial sums (one slot of d for each
    of up to 456 CTAs and each head) and 2048 words of per-head counters: more than the array
    holds.  The call gets real device tensors of the right size (about 150 MiB), so even
    a launch by mistake would stay inside its buffers; it must return SAGE_ERR_WORKSPACE, and the
    partials-needed query must agree."""
    from bit_trainable_attention_sage_gb300 import build
    build.build()
    import bit_trainable_attention_sage_gb300 as sg
    L = sg.lib()
    cap = L.sage_quantize_noalloc_max_partials()
    assert cap == 131072
    B, H, N, d = 1, 2048, 64, 128
    p = sg.make_params(B, H, N, d, sg.binding.SAGE_FP16, False)
    assert L.sage_quantize_noalloc_partials_needed(ctypes.byref(p)) == (456 + B * H) * d + B * H > cap
    Q, K, V = (torch.zeros((B, H, N, d), dtype=torch.float16, device="cuda") for _ in range(3))
    with pytest.raises(sg.binding.SageError) as e:
        sg.sage_quantize_smooth_noalloc(Q, K, V)
    assert e.value.status == sg.binding.SAGE_ERR_WORKSPACE
    assert sg.sage_device_status() == 0
