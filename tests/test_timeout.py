"""A bounded wait that runs out: the prefill kernel's key producer withholds
each CTA's first key tile (FA_DEBUG_WITHHOLD, test only), so the waits behind
it give up after their bound.  The call must report FA_ERR_DEVICE_TIMEOUT in
the workspace, every role must stop and release TMEM, and the context must
stay usable: the next call is checked against the oracle."""
import pytest

import workloads as W
from parity_util import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def test_prefill_wait_runs_out_and_the_context_recovers():
    import torch
    import masked_flash_attention_gb300 as fa
    from parity_util import DEV, to_dev
    c = W.random_case(1600, B=1, Sq=256, Sk=256, Hq=2, Hkv=2, d=128, causal=True)
    p = to_dev(c["params"])
    rc, plan = fa.fa_fwd_plan(c["q"], c["k"], c["v"], **c["params"])
    assert rc == 0 and plan["path"] == fa._lib.FA_PATH_PREFILL
    out, lse, ws = fa.fa_fwd(c["q"].to(DEV), c["k"].to(DEV), c["v"].to(DEV), debug_flags=fa.FA_DEBUG_WITHHOLD, **p)
    torch.cuda.synchronize()
    status, info = fa.fa_check_device_error(ws)
    assert status == fa._lib.FA_ERR_DEVICE_TIMEOUT, (status, info)
    # the context is usable: the same call without the flag matches the oracle
    out2, lse2, _ = run_gpu(c)
    ref_o, ref_l = run_oracle(c)
    compare(out2, lse2, ref_o, ref_l, "after a timed-out call")
