"""Failure detection on the GPU without a fault: every pipeline wait is
bounded, so a wait that nothing satisfies ends with MOK_ERR_TIMEOUT in the
status word and the context stays usable."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import BF16_TOL, assert_close, host, mok
from routing_grouped_expert_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    return mok()


def test_bounded_waits_report_timeout_and_context_survives(m):
    assert m.get_error() == m.MOK_OK
    m.check_wait_timeout()
    assert m.get_error() == m.MOK_ERR_TIMEOUT
    assert m.get_error() == m.MOK_OK  # read and cleared
    # the device keeps working: a forward pass after the expired waits
    cfg = W.CONFIGS["tiny"]
    inp = W.make_inputs(cfg, "cpu")
    d = {k: v.to(DEV) for k, v in inp.items()}
    shape = m.shape_of(cfg)
    ws = torch.empty(m.workspace_bytes(shape, m.OP_FWD), dtype=torch.uint8, device=DEV)
    out = torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16, device=DEV)
    m.moe_fwd(shape, m.make_weights(d), d["x"], d["s"], out, ws)
    m.check_device_status()
    ref = O.moe_forward(host(inp), cfg.K)
    assert_close(out.float().cpu().numpy(), ref["out"], BF16_TOL, "out")
