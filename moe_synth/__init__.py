"""Seeded synthetic inputs for the DeepSeekMoE layer.

This module only draws random numbers and arranges them in the layouts the
layer takes; it holds none of the layer's arithmetic.  Both the CUDA
library's callers and the CPU oracle take their inputs from here.

Workloads (shapes of the DeepSeek-V3 Technical Report, model
hyper-parameters paragraph, scaled where noted):

  tiny_fp32   T=64,   d=256,  E=16  (4 groups, keep 2), K=2, 1 shared, I=128,  fp32
  mid_bf16    T=4096, d=2048, E=64  (8 groups, keep 4), K=6, 2 shared, I=1408, bf16
  v3_bf16     T=8192, d=7168, E=256 (8 groups, keep 4), K=8, 1 shared, I=2048, bf16,
              route scale 2.5, router skewed towards a Zipf(1.1) popularity
  v3_fp8      the v3 shape with FP8 E4M3 expert GEMMs; 72 outlier channels x20
  v3_decode   T=128 decode batch of the v3 shape, bf16, unskewed router

Values: x ~ N(0, 1); expert and shared weights ~ N(0, 0.02); router
centroids ~ N(0, 0.02) (or the skewed construction below); bias 0, except
tiny_fp32 where b ~ U(-0.1, 0.1).

Skewed router: e_i = sigma_i q_i with q_i orthonormal rows (QR of a seeded
Gaussian), so that the logits x . e_i are independent N(0, sigma_i^2); the
per-expert sigma comes from ``zipf_sigma_<name>.txt``, written once by
``calibrate_zipf.py``.

Tensors for a given seed depend on the device they are drawn on (the CPU
and CUDA generators differ); callers that need both a device and a host
copy draw once and copy.
"""

from __future__ import annotations

import os
from dataclasses import dataclass, field, asdict

import torch

HERE = os.path.dirname(os.path.abspath(__file__))


@dataclass(frozen=True)
class LayerShape:
    name: str
    T: int
    d: int
    E: int
    n_groups: int
    topk_groups: int
    k: int
    n_shared: int
    inter: int
    route_scale: float
    gamma: float
    dtype: str            # "fp32" | "bf16" | "fp8"
    seed: int
    bias_init: str = "zero"          # "zero" | "uniform0.1"
    router: str = "gaussian"         # "gaussian" | "zipf"
    outlier_channels: int = 0
    outlier_scale: float = 20.0
    bias_steps: int = 0
    group_score_topn: int = 2

    def as_dict(self):
        return asdict(self)


CONFIGS = {
    "tiny_fp32": LayerShape("tiny_fp32", 64, 256, 16, 4, 2, 2, 1, 128, 1.0, 1e-3,
                            "fp32", 1, bias_init="uniform0.1"),
    "mid_bf16": LayerShape("mid_bf16", 4096, 2048, 64, 8, 4, 6, 2, 1408, 1.0, 1e-3,
                           "bf16", 2),
    "v3_bf16": LayerShape("v3_bf16", 8192, 7168, 256, 8, 4, 8, 1, 2048, 2.5, 1e-3,
                          "bf16", 3, router="zipf", bias_steps=50),
    "v3_fp8": LayerShape("v3_fp8", 8192, 7168, 256, 8, 4, 8, 1, 2048, 2.5, 1e-3,
                         "fp8", 4, router="zipf", outlier_channels=72),
    "v3_decode": LayerShape("v3_decode", 128, 7168, 256, 8, 4, 8, 1, 2048, 2.5, 1e-3,
                            "bf16", 5),
}


def shape_with(base: LayerShape, **kw) -> LayerShape:
    """A copy of ``base`` with some fields replaced (for reduced test cases)."""
    d = base.as_dict()
    d.update(kw)
    return LayerShape(**d)


def storage_dtype(shape: LayerShape):
    """Storage type of x and of the master weights."""
    return torch.float32 if shape.dtype == "fp32" else torch.bfloat16


def zipf_sigma(name="v3"):
    """Per-expert logit scale of the skewed router (256 values)."""
    path = os.path.join(HERE, f"zipf_sigma_{name}.txt")
    vals = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(float(line))
    return torch.tensor(vals, dtype=torch.float64)


def orthonormal_rows(n, d, seed):
    """n orthonormal rows of length d (QR of a seeded Gaussian, on the CPU)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    a = torch.randn(d, n, generator=g, dtype=torch.float64)
    q, r = torch.linalg.qr(a)
    q = q * torch.sign(torch.diagonal(r))[None, :]
    return q.T.contiguous()


def _gen(device, seed):
    return torch.Generator(device=device).manual_seed(seed)


def make_layer(shape: LayerShape, device="cpu", weights=True):
    """Draw one layer's inputs and weights.

    Returns a dict: x [T, d]; router_w [E, d] fp32; bias [E] fp32;
    w13 [E, 2I, d] (rows [0, I) gate W1, rows [I, 2I) up W3); w2 [E, d, I];
    ws13 [Ns, 2I, d]; ws2 [Ns, d, I]; master weights in bf16 (fp32 for
    the fp32 shape).  With ``weights=False`` the expert weights are left
    out (routing-only cases)."""
    dev = torch.device(device)
    g = _gen(dev, shape.seed)
    sd = storage_dtype(shape)
    T, d, E, inter, ns = shape.T, shape.d, shape.E, shape.inter, shape.n_shared
    x = torch.randn(T, d, generator=g, device=dev, dtype=torch.float32)
    if shape.outlier_channels:
        gc = torch.Generator(device="cpu").manual_seed(shape.seed + 1000)
        ch = torch.randperm(d, generator=gc)[: shape.outlier_channels].to(dev)
        x[:, ch] *= shape.outlier_scale
    x = x.to(sd)
    if shape.router == "zipf":
        sigma = zipf_sigma("v3")
        assert sigma.numel() == E
        q = orthonormal_rows(E, d, shape.seed + 2000)
        router_w = (q * sigma[:, None]).to(torch.float32).to(dev)
    else:
        router_w = torch.randn(E, d, generator=g, device=dev, dtype=torch.float32) * 0.02
    if shape.bias_init == "uniform0.1":
        bias = (torch.rand(E, generator=g, device=dev, dtype=torch.float32) * 0.2 - 0.1)
    else:
        bias = torch.zeros(E, device=dev, dtype=torch.float32)
    out = {"x": x.contiguous(), "router_w": router_w.contiguous(), "bias": bias.contiguous()}
    if not weights:
        return out
    w13 = torch.empty(E, 2 * inter, d, device=dev, dtype=sd)
    w2 = torch.empty(E, d, inter, device=dev, dtype=sd)
    for e in range(E):
        w13[e] = (torch.randn(2 * inter, d, generator=g, device=dev, dtype=torch.float32) * 0.02).to(sd)
        w2[e] = (torch.randn(d, inter, generator=g, device=dev, dtype=torch.float32) * 0.02).to(sd)
    ws13 = torch.empty(ns, 2 * inter, d, device=dev, dtype=sd)
    ws2 = torch.empty(ns, d, inter, device=dev, dtype=sd)
    for s in range(ns):
        ws13[s] = (torch.randn(2 * inter, d, generator=g, device=dev, dtype=torch.float32) * 0.02).to(sd)
        ws2[s] = (torch.randn(d, inter, generator=g, device=dev, dtype=torch.float32) * 0.02).to(sd)
    out.update(w13=w13, w2=w2, ws13=ws13, ws2=ws2)
    return out


def make_tokens(shape: LayerShape, n_tokens, device="cpu", seed_offset=0):
    """Extra token batches of the same distribution (e.g. for calibration)."""
    g = _gen(torch.device(device), shape.seed + 7919 + seed_offset)
    return torch.randn(n_tokens, shape.d, generator=g, device=device, dtype=torch.float32)


def make_grad(shape: LayerShape, device="cpu"):
    """Gradient of a loss with respect to the layer output, dL/dy [T, d]:
    standard normal values in the storage type (seeded per shape)."""
    g = _gen(torch.device(device), shape.seed + 5003)
    dy = torch.randn(shape.T, shape.d, generator=g, device=device, dtype=torch.float32)
    return dy.to(storage_dtype(shape)).contiguous()
