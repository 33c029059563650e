"""Host-side checks of the torch.optim-style wrapper that need no GPU."""

import pytest
import torch

from amsgrad_optimizer_step_gb300.optim import FusedAdamW, GradScaler


def test_cpu_parameters_fail_loudly():
    """There is no CPU path: CPU parameters are rejected, not updated some other way."""
    with pytest.raises(ValueError, match="CUDA parameters"):
        FusedAdamW([torch.nn.Parameter(torch.zeros(3))])


@pytest.mark.parametrize("kwargs,match", [
    ({"fused_step": False}, "fused step only"),
    ({"max_grad_norm": 0.0}, "max_grad_norm"),
    ({"max_grad_norm": -1.0}, "max_grad_norm"),
])
def test_invalid_options_are_rejected_before_any_bucket(kwargs, match):
    with pytest.raises(ValueError, match=match):
        FusedAdamW([torch.nn.Parameter(torch.zeros(3))], **kwargs)


def test_grad_scaler_schedule():
    """Backs off by half after a skipped step, grows after growth_interval clean ones."""
    class _Opt:
        def __init__(self):
            self.last_report = {}
            self.skips = [False, True, False, False, False]

        def step(self, gradient_scale, check_finite):
            assert check_finite
            self.last_report = {"skipped": self.skips.pop(0)}

    opt = _Opt()
    sc = GradScaler(init_scale=1024.0, growth_interval=3)
    scales = []
    for _ in range(5):
        sc.step(opt)
        sc.update()
        scales.append(sc.get_scale())
    assert scales == [1024.0, 512.0, 512.0, 512.0, 1024.0]
    sd = sc.state_dict()
    other = GradScaler()
    other.load_state_dict(sd)
    assert other.get_scale() == 1024.0 and other.state_dict() == sd
