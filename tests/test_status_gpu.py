"""The device status word: a bounded wait that runs out is reported, and the
context stays usable.

No fault, trap or endless wait is involved. The plan option debug_stall makes
the tcgen05 PAC's MMA thread wait (for about a millisecond) on a barrier that
nothing arrives on before it issues anything. The other roles of each block
then meet their own bounded waits, drain the TMA loads they issued and leave;
the kernels return, pst_plan_check_status reports the timeout bit, and a
normal call right after gives the oracle's result."""
import numpy as np
import pytest

import synth
from oracle import attention as oa

pytestmark = pytest.mark.gpu

ABS_TOL, LSE_TOL = 2e-3, 1e-3
WAIT_TIMEOUT_BIT = 1


@pytest.mark.parametrize("n_req", [64, 16], ids=["rows256", "rows64"])
def test_wait_that_runs_out_is_reported_and_next_call_is_clean(lib, n_req):
    import torch
    from prefix_shared_tree_gb300.torch_api import TreeDecodeAttention, to_device
    wl = synth.document_qa(prefix=1024, n_req=n_req)
    K, V = wl.kv_pools()
    Q = wl.q()
    Qd, Kd, Vd = to_device(Q, wl.dtype), to_device(K, wl.dtype), to_device(V, wl.dtype)
    stalled = TreeDecodeAttention.from_workload(wl, debug_stall=True)
    assert stalled.plan.stats()["n_tc_items"] > 0
    stalled(Qd, Kd, Vd)
    torch.cuda.synchronize()
    code = stalled.check_status()
    assert code & WAIT_TIMEOUT_BIT, f"status word {code}"
    assert stalled.check_status() == 0, "reading the status word clears it"
    # the context is usable and a normal plan gives the oracle's result
    normal = TreeDecodeAttention.from_workload(wl)
    O, L = normal(Qd, Kd, Vd)
    torch.cuda.synchronize()
    assert normal.check_status() == 0
    Oref, Lref = oa.decode_attention(wl, K, V, Q)
    assert np.abs(O.cpu().numpy() - Oref).max() <= ABS_TOL
    assert np.abs(L.cpu().numpy() - Lref).max() <= LSE_TOL
