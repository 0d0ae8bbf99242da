"""The five workloads at their full sizes, through the C ABI in the launch configuration bench.py
times, compared element by element with the CPU oracle on the same seeded inputs (O and the final
W_down against the bounds 1e-4 fp32 / 2e-2 bf16, plus the fast-part diagnostics).  The oracle runs
in float64 on the host cores: about 1-15 TFLOP of work per workload."""
import json
import os

import pytest
import torch

from tests.util import layer_check, to_dev
from weight_mlp_layers_swiglu_b300.inputs import WORKLOAD_ORDER, WORKLOADS, make_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def ctx():
    import weight_mlp_layers_swiglu_b300 as pkg

    c = pkg.Context(0)
    yield c
    c.close()


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_full_size_workload(ctx, name):
    w = WORKLOADS[name]
    x = make_inputs(w)
    xd = to_dev(x)
    O, Wf = ctx.layer_forward(xd["H"], xd["X0"], xd["W_gate"], xd["W_up"], xd["W_down0"], xd["W_target"],
                              xd["conv_w"], w.C, w.eta)
    assert ctx.sync() == 0, ctx.last_error()
    O, Wf = O.cpu(), Wf.cpu()
    del xd
    ctx._ws = None
    torch.cuda.empty_cache()
    errs = layer_check(w, x, O, Wf)
    out = os.environ.get("IPTTT_RESULTS_DIR")  # optional: a directory for the measured errors
    if out and os.path.isdir(out):
        with open(os.path.join(out, f"parity_{name}.json"), "w") as f:
            json.dump({"workload": name, **errs}, f)
    print(name, errs)
