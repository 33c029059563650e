"""The five seeded workloads, as plain data plus their input recipes.

Each workload fixes the element count (and, for the decoder-shaped bucket, the
tensor layout), the gradient storage type, the hyper-parameters and the
per-call controls.  Inputs are produced by ``synthetic.generators`` so that the
host (numpy, any sampled index) and the device (torch, in chunks) agree bit for
bit.  Nothing here computes any part of the optimizer.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

from . import generators as G

F32, F16, BF16 = "f32", "f16", "bf16"

STREAM_PARAM = 1
STREAM_GRAD = 2
STREAM_OUTLIER = 3


def decoder_bucket_shapes() -> list[tuple[str, tuple[int, ...]]]:
    """Tensor shapes of the 1.1B-parameter decoder bucket, in bucket order."""
    shapes = [("embed", (32000, 2048))]
    for layer in range(22):
        for name in ("q", "k", "v", "o"):
            shapes.append((f"l{layer}.{name}", (2048, 2048)))
        shapes.append((f"l{layer}.gate", (5632, 2048)))
        shapes.append((f"l{layer}.up", (5632, 2048)))
        shapes.append((f"l{layer}.down", (2048, 5632)))
        shapes.append((f"l{layer}.norm_attn", (2048,)))
        shapes.append((f"l{layer}.norm_mlp", (2048,)))
    return shapes


def decoder_bucket_offsets() -> np.ndarray:
    """Segment boundaries (nseg + 1 entries) of the decoder bucket."""
    sizes = [int(np.prod(s)) for _, s in decoder_bucket_shapes()]
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n: int
    grad_dtype: str
    seed: int
    calls: int
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-5
    weight_decay: float = 1e-4
    amsgrad: bool = False
    maximize: bool = False
    gradient_scale: float = 1.0
    param_sigma: float = 0.02
    grad_sigma: float = 1e-2
    grad_premul: float = 1.0            # FP32 factor applied before rounding (x128 case)
    outlier_per_10000: int = 0          # Bernoulli mask rate, in 1/10000
    outlier_mult: float = 1.0
    skip_calls: tuple[int, ...] = ()    # 1-based call indices with skip_update = true
    inf_call: Optional[int] = None      # 1-based call whose gradient holds one planted value
    inf_value: float = float("inf")     # the planted value (+Inf, or a large finite one)
    inplace: bool = False
    row_len: int = 0                    # > 0: analyze rows of this length
    max_grad_norm: float = 0.0          # > 0: global L2 clip
    segments: Optional[tuple[int, ...]] = None   # bucket segment boundaries

    # ---- derived -------------------------------------------------------
    def scaled(self, n: int, **changes) -> "Workload":
        """Same recipe at a different size (a single flat segment)."""
        return dataclasses.replace(self, n=n, segments=None, **changes)

    @property
    def grad_bytes(self) -> int:
        return 4 if self.grad_dtype == F32 else 2

    def inf_index(self) -> int:
        """Index that holds +Inf in call ``inf_call`` (drawn from numpy's PCG64 with the seed)."""
        return int(np.random.default_rng(self.seed).integers(self.n))

    def options(self) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay, amsgrad=self.amsgrad,
                    maximize=self.maximize)

    # ---- host inputs at arbitrary indices --------------------------------
    def params_host(self, idx) -> np.ndarray:
        return G.normal_np(idx, self.param_sigma, G.stream_key(self.seed, STREAM_PARAM))

    def grad_f32_host(self, call: int, idx) -> np.ndarray:
        idx = np.asarray(idx, dtype=np.int64)
        x = G.normal_np(idx, self.grad_sigma, G.stream_key(self.seed, STREAM_GRAD, call))
        if self.grad_premul != 1.0:
            x = x * np.float32(self.grad_premul)
        if self.outlier_per_10000:
            mask = G.bernoulli_np(idx, self.outlier_per_10000,
                                  G.stream_key(self.seed, STREAM_OUTLIER, call))
            x = np.where(mask, x * np.float32(self.outlier_mult), x).astype(np.float32)
        if self.inf_call is not None and call == self.inf_call:
            x = np.where(idx == self.inf_index(), np.float32(self.inf_value), x).astype(np.float32)
        return x

    def grad_host(self, call: int, idx) -> np.ndarray:
        """Stored gradient at ``idx`` for 1-based ``call``: float32, or uint16 bits."""
        x = self.grad_f32_host(call, idx)
        if self.grad_dtype == F32:
            return x
        if self.grad_dtype == BF16:
            return G.f32_to_bf16_bits_np(x)
        return G.f32_to_f16_bits_np(x)

    # ---- device inputs ---------------------------------------------------
    def fill_params_device(self, out, chunk: int = 1 << 25) -> None:
        for s in range(0, self.n, chunk):
            c = min(chunk, self.n - s)
            out[s:s + c].copy_(G.normal_torch(s, c, self.param_sigma,
                                              G.stream_key(self.seed, STREAM_PARAM), out.device))

    def fill_grad_device(self, call: int, out, chunk: int = 1 << 25) -> None:
        """Write the stored gradient of ``call`` into ``out`` (float32/float16/bfloat16)."""
        import torch
        for s in range(0, self.n, chunk):
            c = min(chunk, self.n - s)
            x = G.normal_torch(s, c, self.grad_sigma,
                               G.stream_key(self.seed, STREAM_GRAD, call), out.device)
            if self.grad_premul != 1.0:
                x.mul_(torch.tensor(self.grad_premul, dtype=torch.float32, device=out.device))
            if self.outlier_per_10000:
                mask = G.bernoulli_torch(s, c, self.outlier_per_10000,
                                         G.stream_key(self.seed, STREAM_OUTLIER, call), out.device)
                x = torch.where(mask, x * torch.tensor(self.outlier_mult, dtype=torch.float32,
                                                       device=out.device), x)
            if self.inf_call is not None and call == self.inf_call:
                k = self.inf_index()
                if s <= k < s + c:
                    x[k - s] = float(np.float32(self.inf_value))
            if self.grad_dtype == F32:
                out[s:s + c].copy_(x)
            elif self.grad_dtype == BF16:
                G.store_bits_torch(G.f32_to_bf16_bits_torch(x), out[s:s + c])
            else:
                out[s:s + c].copy_(x.to(torch.float16))


CONFIG1 = Workload(name="flat65536_f32", n=65_536, grad_dtype=F32, seed=0, calls=10,
                   weight_decay=1e-4)

CONFIG2 = Workload(name="flat65537_bf16x128_amsgrad", n=65_537, grad_dtype=BF16, seed=1,
                   calls=20, weight_decay=0.01, amsgrad=True, gradient_scale=128.0,
                   grad_premul=128.0, skip_calls=(5,))

CONFIG3 = Workload(name="flat124M_bf16_outliers_inplace", n=124_439_808, grad_dtype=BF16,
                   seed=2, calls=50, weight_decay=0.01, grad_sigma=1e-3,
                   outlier_per_10000=100, outlier_mult=100.0, inplace=True)

_OFF4 = tuple(int(x) for x in decoder_bucket_offsets())
CONFIG4 = Workload(name="decoder1.1B_bucket_f16_amsgrad", n=_OFF4[-1], grad_dtype=F16,
                   seed=3, calls=10, amsgrad=True, grad_sigma=1e-3, inplace=True,
                   segments=_OFF4)
CONFIG4_MAX = dataclasses.replace(CONFIG4, name="decoder1.1B_bucket_f16_amsgrad_maximize",
                                  maximize=True)

CONFIG5 = Workload(name="flat1G_bf16_stats_clip", n=1_073_741_824, grad_dtype=BF16, seed=4,
                   calls=5, grad_sigma=1e-3, inf_call=3, inplace=True, row_len=256,
                   max_grad_norm=1.0)

ALL = (CONFIG1, CONFIG2, CONFIG3, CONFIG4, CONFIG4_MAX, CONFIG5)
