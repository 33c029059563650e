"""The shared-memory pipeline's bounded waits give up cleanly (no fault, no hang).

fa_pipeline_selftest launches one steady update whose stage barriers wait for
16 bytes that are never sent.  Every wait must run out after its limit, the
kernel must set the device flag, drain its own copies and return without
writing p, m or v, and the context must stay usable for the next real step.
"""

import time

import numpy as np
import pytest
import torch

import amsgrad_optimizer_step_gb300 as fa
import oracle
from gpu_harness import gate

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from amsgrad_optimizer_step_gb300 import build
    build.build()


def test_bounded_waits_give_up_cleanly(oracle_lib):
    n = 4_000_003
    gen = torch.Generator(device=DEV).manual_seed(7)
    p = torch.randn(n, device=DEV, generator=gen) * 0.02
    m = torch.randn(n, device=DEV, generator=gen) * 1e-3
    v = torch.rand(n, device=DEV, generator=gen) * 1e-6
    g = (torch.randn(n, device=DEV, generator=gen) * 1e-2).to(torch.bfloat16)
    snap = [x.clone() for x in (p, m, v)]
    assert fa.fa_device_error(clear=True) == 0
    t0 = time.perf_counter()
    flag = fa.fa_pipeline_selftest(p, g, m, v)
    elapsed = time.perf_counter() - t0
    assert flag == 1, "the waits did not give up"
    assert elapsed < 60.0
    for a, b in zip((p, m, v), snap):
        assert torch.equal(a, b), "a pipeline that gave up wrote its outputs"
    assert fa.fa_device_error() == 0  # the self-test cleared its flag

    # the context is still usable: a real step matches the oracle
    opts = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=1e-4, amsgrad=False,
                maximize=False)
    idx = np.random.default_rng(8).integers(0, n, 5000)
    before = [x[torch.as_tensor(idx, device=DEV)].double().cpu().numpy() for x in (p, m, v)]
    gbits = g.view(torch.int16)[torch.as_tensor(idx, device=DEV)].cpu().numpy().view(np.uint16)
    t, upd = fa.fa_adamw_step_inplace(p, g, m, v, None, 5, fa.options(**opts), fa.control())
    torch.cuda.synchronize()
    assert upd and t == 6 and fa.fa_device_error() == 0
    ref = [np.array(b) for b in before] + [np.zeros(len(idx))]
    oracle_lib.update(gbits, "bf16", opts, 1.0, 1.0, 6, True, True, *ref)
    gate(p[torch.as_tensor(idx, device=DEV)].cpu().numpy(), ref[0], 1e-6, "p after self-test")


def test_selftest_needs_the_shared_memory_path():
    n = 1000
    p, m, v = (torch.zeros(n, device=DEV) for _ in range(3))
    g = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fa.FusedAdamWError) as e:
        fa.fa_pipeline_selftest(p, g, m, v)
    assert e.value.status == 3
