"""The bounded device waits: a wait that nothing will satisfy ends with SAGE_ERR_TIMEOUT, and
the GPU stays usable.

A test-only copy of the library (build variant "faultsim": waits give up after 2e8 cycles,
about 0.1 s, and the backward's TMA producer never issues the Q^ block of step 1) runs one
backward.  Its MMA thread waits for that block, gives up, and raises the CTA's abort flag.  Every
other wait of the CTA then returns at once.  The score warps leave their loop together at the
tile-maximum barrier.  The producers drain the copies they issued and the MMA thread the MMAs it
committed, so the kernel exits and sage_device_status() reports SAGE_ERR_TIMEOUT.  The same
process then runs the product library end to end and must get SAGE_OK and finite results.

The run happens in a child process with its own time limit, so a mistake in the abort path
shows up as a failed test rather than a hung one.
"""
import json
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import ctypes, json, sys, time
    sys.path.insert(0, ROOT)
    import torch
    import bit_trainable_attention_sage_gb300 as sg
    from bit_trainable_attention_sage_gb300 import build
    fs = ctypes.CDLL(build.build(variant="faultsim"))
    P = ctypes.POINTER(sg.SageParams)
    vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    for name in ("sage_quantize_workspace_bytes", "sage_fwd_workspace_bytes", "sage_bwd_workspace_bytes"):
        getattr(fs, name).argtypes = [P]; getattr(fs, name).restype = sz
    fs.sage_quantize_smooth.argtypes = [P] + [vp] * 12 + [sz, vp]
    fs.sage_attn_fwd.argtypes = [P] + [vp] * 12 + [sz, vp]
    fs.sage_attn_bwd.argtypes = [P] + [vp] * 15 + [sz, vp]
    fs.sage_device_status.argtypes = [vp]
    B, H, N, d = 1, 2, 256, 128
    g = torch.Generator().manual_seed(0)
    Q, K, V, dO = (torch.randn((B, H, N, d), generator=g).half().cuda() for _ in range(4))
    p = sg.make_params(B, H, N, d, 0, False)
    st = torch.cuda.current_stream().cuda_stream
    i8 = lambda: torch.empty((B, H, N, d), dtype=torch.int8, device="cuda")
    f32 = lambda *s: torch.empty(s, dtype=torch.float32, device="cuda")
    Qh, Kh, Vh = i8(), i8(), i8()
    sQ, sK, sV = f32(B, H, N // 64), f32(B, H, N // 64), f32(B, H, N // 64)
    muK = f32(B, H, d)
    ws = lambda q: torch.empty(max(q(ctypes.byref(p)), 16), dtype=torch.uint8, device="cuda")
    wq, wf, wb = ws(fs.sage_quantize_workspace_bytes), ws(fs.sage_fwd_workspace_bytes), ws(fs.sage_bwd_workspace_bytes)
    O = torch.empty((B, H, N, d), dtype=torch.float16, device="cuda")
    L = f32(B, H, N)
    dQ, dK, dV = f32(B, H, N, d), f32(B, H, N, d), f32(B, H, N, d)
    ptr = lambda t: None if t is None else t.data_ptr()
    rc = [fs.sage_quantize_smooth(ctypes.byref(p), *map(ptr, (Q, K, V, Qh, Kh, Vh, sQ, sK, sV, muK, None, wq)),
                                  wq.numel(), st)]
    rc.append(fs.sage_attn_fwd(ctypes.byref(p), *map(ptr, (Qh, Kh, Vh, sQ, sK, sV, None, None, None, O, L, wf)),
                               wf.numel(), st))
    fwd_status = fs.sage_device_status(st)
    t0 = time.time()
    rc.append(fs.sage_attn_bwd(ctypes.byref(p), *map(ptr, (Qh, Kh, sQ, sK, None, None, None, V, O, L, dO, dQ, dK, dV, wb)),
                               wb.numel(), st))
    bwd_status = fs.sage_device_status(st)
    secs = time.time() - t0
    # the product library, same process and device: the context must still work
    q = sg.sage_quantize_smooth(Q, K, V)
    O2, L2 = sg.sage_attn_fwd(q, causal=False)
    g2 = sg.sage_attn_bwd(q, V, O2, L2, dO, causal=False)
    ok_status = sg.sage_device_status()
    finite = bool(all(torch.isfinite(t).all().item() for t in g2))
    print(json.dumps(dict(rc=rc, fwd_status=fwd_status, bwd_status=bwd_status, seconds=secs,
                          after_status=ok_status, finite=finite)))
""").replace("ROOT", repr(ROOT))


def test_backward_wait_that_never_completes_reports_timeout():
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    print("\n", out)
    assert out["rc"] == [0, 0, 0]
    assert out["fwd_status"] == 0                     # the forward has no skipped copy
    assert out["bwd_status"] == 5                     # SAGE_ERR_TIMEOUT
    assert out["seconds"] < 30
    assert out["after_status"] == 0 and out["finite"]
