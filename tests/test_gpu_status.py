"""Failure detection without a GPU fault: a bounded device-side wait that runs
out records MOE_ERR_DEVICE_TIMEOUT in the workspace status word, the host reads
it, and the context stays usable for the next kernels."""
import numpy as np
import pytest
import torch

from grouped_gemm_moe_gb300 import binding as B

from _parity import dev, ensure_built

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    ensure_built()
    ws = B.new_workspace(B.WORKSPACE_HEADER, dev())
    assert B.moe_read_device_status(ws) == 0
    B.moe_debug_wait_timeout(ws, 20000)            # 20 ms limit on a barrier nothing completes
    assert B.moe_read_device_status(ws) == B.MOE_ERR_DEVICE_TIMEOUT
    assert B.moe_read_device_status(ws) == 0       # reading clears the word
    # the context is still usable: a grouped GEMM runs and reports no error
    g = torch.Generator(device=dev()).manual_seed(0)
    E, d, I, M = 2, 128, 128, 300
    off = torch.tensor([0, 100, M], dtype=torch.int32, device=dev())
    xp = torch.randn(M, d, device=dev(), generator=g).to(torch.bfloat16)
    w = [(torch.randn(E, a, b, device=dev(), generator=g) * 0.02).to(torch.bfloat16)
         for a, b in ((d, I), (d, I), (I, d))]
    ws2 = B.new_workspace(B.WORKSPACE_HEADER, dev())
    y, h, gu = B.moe_grouped_ffn(xp, off, *w, ws=ws2)
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws2) == 0
    assert torch.isfinite(y.float()).all()
