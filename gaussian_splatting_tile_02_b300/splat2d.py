"""2D splats on the tile pipeline (gs_rasterize_2d / gs_rasterize_2d_backward).

The lesson page "3D Gaussian Splatting à partir de zéro":
- section "Étape 2": ``rasterise_2d``, Gaussians given directly in image space,
  composited front to back in the order of a learned per-Gaussian scalar;
- section "Étape 3": a trainable 2D scene, with a mean, a log-scale pair, a
  rotation angle, colour and opacity logits and that ordering scalar per
  Gaussian;
- section "Étape 4": fitting it to a target image by gradient descent on the
  mean squared error.

``rasterise_2d`` is a ``torch.autograd.Function`` whose forward and backward
are the library's CUDA kernels (binning, radix sorts, compositing and its
backward are those of the 3D renderer). ``Splats2D`` and ``fit`` are a small
model and training loop on top of it: the activations (rotation and scales to
a covariance, sigmoids) are the model's, in PyTorch autograd, and the
optimiser is ``torch.optim.Adam``.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np

from .native import check, lib


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream():
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def key_capacity(n: int, width: int, height: int) -> int:
    """Upper bound on the (Gaussian, tile) pairs: every Gaussian on every tile."""
    return int(n) * ((int(width) + 15) // 16) * ((int(height) + 15) // 16)


def _forward(means, covs, colours, opacities, depths, height: int, width: int):
    torch = _torch()
    n = int(means.shape[0])
    cap = key_capacity(n, width, height)
    wsb = int(lib().gs_render_workspace_bytes(n, width, height, cap))
    dev = means.device
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    image = torch.empty((height, width, 3), dtype=torch.float32, device=dev)
    final_T = torch.empty((height, width), dtype=torch.float32, device=dev)
    n_contrib = torch.empty((height, width), dtype=torch.int32, device=dev)
    check(lib().gs_rasterize_2d(_ptr(means), _ptr(covs), _ptr(colours), _ptr(opacities), _ptr(depths), n, width,
                                height, cap, _ptr(ws), wsb, _ptr(image), _ptr(final_T), _ptr(n_contrib), _stream()),
          "gs_rasterize_2d")
    return image, final_T, n_contrib, ws, cap


def _make_function():
    torch = _torch()

    class Rasterise2D(torch.autograd.Function):
        @staticmethod
        def forward(ctx, means, covs, colours, opacities, depths, height, width):
            c = lambda t: t.detach().to(torch.float32).contiguous()
            m, cv, co, op, dp = c(means), c(covs), c(colours), c(opacities), c(depths)
            image, final_T, n_contrib, ws, cap = _forward(m, cv, co, op, dp, int(height), int(width))
            ctx.save_for_backward(cv, final_T, n_contrib, ws)
            ctx.dims = (int(m.shape[0]), int(height), int(width), cap)
            return image

        @staticmethod
        def backward(ctx, grad_image):
            cv, final_T, n_contrib, ws = ctx.saved_tensors
            n, height, width, cap = ctx.dims
            dev = cv.device
            gm = torch.empty((n, 2), dtype=torch.float32, device=dev)
            gc = torch.empty((n, 2, 2), dtype=torch.float32, device=dev)
            gco = torch.empty((n, 3), dtype=torch.float32, device=dev)
            go = torch.empty(n, dtype=torch.float32, device=dev)
            gi = grad_image.to(torch.float32).contiguous()
            check(lib().gs_rasterize_2d_backward(_ptr(cv), n, width, height, cap, _ptr(ws), ws.numel(),
                                                 _ptr(final_T), _ptr(n_contrib), _ptr(gi), _ptr(gm), _ptr(gc),
                                                 _ptr(gco), _ptr(go), _stream()), "gs_rasterize_2d_backward")
            return gm, gc, gco, go, None, None, None

    return Rasterise2D


_FN = None


def rasterise_2d(means, covs, colours, opacities, depths, image_size):
    """Image [H, W, 3] of 2D Gaussians (CUDA tensors): means [G, 2], covs [G, 2, 2],
    colours [G, 3], opacities [G], depths [G] (ordering only; no gradient).
    Differentiable in means, covs, colours and opacities."""
    global _FN
    if _FN is None:
        _FN = _make_function()
    H, W = image_size
    return _FN.apply(means, covs, colours, opacities, depths, int(H), int(W))


def target_image(size: int = 64) -> np.ndarray:
    """The worked example's target: on a black background, a red disc of
    radius 10 centred at (20, 20) and a blue square of half-width 8 centred at
    (45, 40) (pixel coordinates (x, y) at integer points)."""
    y, x = np.mgrid[0:size, 0:size]
    img = np.zeros((size, size, 3), np.float32)
    img[(x - 20) ** 2 + (y - 20) ** 2 < 100] = (1.0, 0.2, 0.2)
    img[(np.abs(x - 45) < 8) & (np.abs(y - 40) < 8)] = (0.2, 0.3, 1.0)
    return img


def _module():
    torch = _torch()
    nn = torch.nn

    class Splats2D(nn.Module):
        """Trainable 2D Gaussians: position, log-scale pair, rotation angle,
        colour and opacity logits, and the scalar that orders them."""

        def __init__(self, num: int = 64, size: int = 64, seed: int = 0):
            super().__init__()
            gen = torch.Generator().manual_seed(seed)
            self.means = nn.Parameter(torch.rand(num, 2, generator=gen) * size)
            self.log_scale = nn.Parameter(torch.full((num, 2), math.log(2.0)))
            self.rot = nn.Parameter(torch.zeros(num))
            self.colour_logits = nn.Parameter(0.5 * torch.randn(num, 3, generator=gen))
            self.opacity_logit = nn.Parameter(torch.zeros(num))
            self.depth = nn.Parameter(torch.rand(num, generator=gen))

        def covs(self):
            c, s = torch.cos(self.rot), torch.sin(self.rot)
            rows = torch.stack([torch.stack([c, -s], -1), torch.stack([s, c], -1)], -2)   # R
            var = torch.exp(2.0 * self.log_scale)                                        # diag(s^2)
            return rows @ torch.diag_embed(var) @ rows.transpose(-1, -2)

        def forward(self, size: int):
            return rasterise_2d(self.means, self.covs(), torch.sigmoid(self.colour_logits),
                                torch.sigmoid(self.opacity_logit), self.depth, (size, size))

    return Splats2D


def Splats2D(num: int = 64, size: int = 64, seed: int = 0):
    return _module()(num, size, seed)


def fit(steps: int = 200, num: int = 64, size: int = 64, lr: float = 0.05, seed: int = 0, device="cuda",
        log_every: int = 0) -> dict:
    """Fits ``num`` Gaussians to ``target_image(size)`` with Adam on the mean
    squared error; returns the per-step losses and the final image."""
    torch = _torch()
    target = torch.tensor(target_image(size), device=device)
    model = Splats2D(num, size, seed).to(device)
    opt = torch.optim.Adam(model.parameters(), lr=lr)
    losses = []
    for step in range(steps):
        pred = model(size)
        loss = torch.mean((pred - target) ** 2)
        opt.zero_grad()
        loss.backward()
        opt.step()
        losses.append(float(loss.detach()))
        if log_every and step % log_every == 0:
            print(f"step {step:4d}  mse {losses[-1]:.5f}")
    with torch.no_grad():
        final = model(size)
    return {"losses": losses, "image": final.detach().cpu().numpy(), "model": model,
            "final_mse": float(torch.mean((final - target) ** 2))}
