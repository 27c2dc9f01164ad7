"""Two routes to the agreement band tau at full size on the workloads' own
inputs (x W_x^T projected on the tensor cores): Newton with one more
iteration than configured (K = 4), and two Picard sweeps followed by K = 3
Newton iterations from their result (FAQs, "How many Newton iterations
should I use?": raise K, or try a Picard warm start).  At the configured K
workloads 1, 2 and 4 miss tau = 1e-4 against the float64 unroll by the
method's own error; both routes reach it.  The oracle builds its inputs from
the same seeded x and W_x (a float64 projection of the sampled units' rows,
rounded to the storage type)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 5e-2}


@pytest.mark.parametrize("wl", [1, 2, 3, 4])
def test_both_routes_reach_tau_against_the_unroll(wl):
    import nonlinear_rnn_gb300 as nr
    w = syn.WORKLOADS[wl]
    inp = syn.make_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    P = nr.input_projection(torch.from_numpy(inp["x"]).cuda().to(tdt),
                            torch.from_numpy(inp["W_x"]).cuda().to(tdt))
    cu = inp["cu_seqlens"]
    units = np.array([0, w.d_h // 3, w.d_h // 2, w.d_h - 1])
    cols = np.concatenate([units, w.d_h + units, 2 * w.d_h + units])
    Pc = oracle.input_projection(inp["x"], inp["W_x"][cols]).astype(np.float32)
    if w.dtype == "bf16":
        Pc = syn.round_bf16(Pc)
    Hs = oracle.sequential(Pc, oracle.pack_params(inp["params"])[:, units], cu_seqlens=cu,
                           threads=4)
    ut = torch.as_tensor(units, device="cuda")
    errs = {}
    for name, kw in (("K4", {"K": 4}), ("picard2_K3", {"K": 3, "picard_iters": 2})):
        H, rho = nr.newton_forward(P, inp["params"], cu_seqlens=cu, check=False, **kw)
        errs[name] = float(np.max(np.abs(H[:, :, ut].double().cpu().numpy() - Hs)))
        assert np.isfinite(rho.item())
    assert errs["K4"] <= TOL[w.dtype], errs
    assert errs["picard2_K3"] <= TOL[w.dtype], errs
