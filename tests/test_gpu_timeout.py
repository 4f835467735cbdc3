"""The relocation kernel's failure path, made to run on purpose without any
fault: every pipeline wait of the kernel is bounded, and the testing hook
kvrp_test_set_wait_limit shortens that bound to a few dozen cycles, far below
the latency of one TMA copy, so the first waits give up.  The launch must then
report KVRP_DEV_TIMEOUT in the status word, drain its copies and tensor-core
work, free its TMEM and return (the call and the synchronisation after it
complete), and the next launch on the same stream, with the default limit,
must be exact against the fp64 oracle.  Nothing here traps, faults or hangs:
the waits that run out are ordinary bounded waits on barriers that do
complete a moment later."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from position_invariant_kv_gb300.build import build
    build()
    import position_invariant_kv_gb300 as kvrp
    kvrp.lib()
    yield
    kvrp.kvrp_test_set_wait_limit(0)


@pytest.mark.parametrize("batch", [False, True], ids=["single", "batch"])
def test_short_wait_limit_reports_timeout_and_the_next_call_is_exact(batch):
    import harness
    import position_invariant_kv_gb300 as kvrp
    from oracle import run_workload
    from oracle.compare import parity_report
    spec = ((700, -4096, 32, 0), (300, 1234, 0, 0)) if batch else ((700, -4096, 32, 0),)
    wl = W.small_gqa(seed=990, n_layers=4, n_heads=4, head_dim=128, chunks_spec=spec, extra_pages=1)
    dwl = harness.DeviceWorkload(wl)
    stream = torch.cuda.current_stream()
    try:
        kvrp.kvrp_test_set_wait_limit(32)
        dwl.run(stream=stream)
    finally:
        kvrp.kvrp_test_set_wait_limit(0)
    torch.cuda.synchronize()                      # the launch returns: it drained and exited
    assert dwl.status_value() & kvrp.KVRP_DEV_TIMEOUT
    dwl.status.zero_()
    dwl.reset_pools()
    dwl.run(stream=stream)                        # the same stream, the default limit
    torch.cuda.synchronize()
    assert dwl.status_value() == 0
    got = dwl.pools_host()
    want, refs, conds = run_workload(wl, dwl.host)
    for name in wl.tensors:
        untouched = np.isnan(refs[name]).all(axis=-1)
        assert np.array_equal(got[name][untouched], want[name][untouched]), name
        r = parity_report(got[name][~untouched], refs[name][~untouched], conds[name][~untouched])
        assert r["violations"] == 0 and r["mismatches"] <= 1e-5 * r["n"] + 2, (name, r)
