"""Small helpers shared by GPU tests."""
import math

import torch


def small_tc_run(T=512, H=2, nseg=4):
    """One forward + backward of a bf16 Dk = Dv = 128 problem (tensor-core path)."""
    from state_summary_scan_gb300 import api
    gen = torch.Generator().manual_seed(5)
    q, k, v, dO = (torch.randn(1, T, H, 128, generator=gen).to(torch.bfloat16).cuda() for _ in range(4))
    g = torch.nn.functional.logsigmoid(torch.randn(1, T, H, generator=gen) + 4).cuda()
    plan = api.plan_like(q, v, nseg, 64, 1 / math.sqrt(128))
    api.forward(plan, q, k, v, g)
    out = api.backward(plan, q, k, v, g, dO)
    torch.cuda.synchronize()
    return out
