"""PyTorch autograd over the C ABI: differentiable projection and backprojection.

The forward projector A and the backprojector A^T of one plan are each other's
gradient (the pair is matched, so d<A x, g>/dx = A^T g and d<A^T y, h>/dy = A h),
which also makes second derivatives -- Hessian-vector products of data losses --
available through ordinary autograd.  Leading batch / channel dimensions loop
over the C calls; every call runs in the CUDA library (diffct's
ProjectorFunction / BackprojectorFunction pair, README "Matched operators":
volume and sinogram gradients and Hessian-vector products; CHANGELOG 2.3.0:
leading batch and channel dimensions, including empty batches).
"""

from __future__ import annotations

import torch

import dataclasses

from ._binding import (Geometry, Plan, Volume, ctp_backward, ctp_forward, ctp_geometry_vjp,
                       ctp_plan, ctp_ramp_filter, ctp_surface_vjp, ctp_weighted_backproject,
                       ctp_weighted_backproject_transpose)


class Projector:
    """A plan plus differentiable ``project`` (A) and ``backproject`` (A^T).

    ``project(vol)``: vol of shape (..., D, H, W) -> sinogram (..., n_views, n_v, n_u).
    ``backproject(sino)``: the transpose.  Inputs are moved to the plan's device
    and made contiguous float32; outputs are float32 on that device.
    """

    def __init__(self, geometry: Geometry, volume: Volume, path: str = "auto"):
        self.plan: Plan = ctp_plan(geometry, volume, path)
        self.device = torch.device("cuda", self.plan.device)

    @property
    def vol_shape(self):
        return self.plan.vol_shape

    @property
    def sino_shape(self):
        return self.plan.sino_shape

    def project(self, vol: torch.Tensor) -> torch.Tensor:
        return _Project.apply(vol, self)

    def backproject(self, sino: torch.Tensor) -> torch.Tensor:
        return _Backproject.apply(sino, self)

    def fdk(self, sino: torch.Tensor, view_weight: torch.Tensor | None = None,
            ramp: str = "ramlak", pixel_weight: torch.Tensor | None = None) -> torch.Tensor:
        """Differentiable FBP / FDK: ramp filter (cosine and view weights) then the
        weighted gather; the gradient is the transposed filter of the gather's
        transpose (diffct README "Differentiable FBP and FDK": sinogram gradients
        through the transposed interpolation stencil).  ``view_weight``: (n_views,)
        tensor, e.g. ``full_scan_view_weights``; no gradient flows to it."""
        vw = pw = None
        if view_weight is not None:
            vw = view_weight.detach().to(device=self.device, dtype=torch.float32).contiguous()
        if pixel_weight is not None:
            pw = pixel_weight.detach().to(device=self.device, dtype=torch.float32).contiguous()
        return _Gather.apply(_Filter.apply(sino, self, vw, ramp, False, pw), self)

    __call__ = project


def _batched(x: torch.Tensor, inner: tuple, name: str):
    if tuple(x.shape[-len(inner):]) != tuple(inner):
        raise ValueError(f"{name} must end with shape {tuple(inner)}, got {tuple(x.shape)}")
    return x.shape[:-len(inner)]


def _apply(proj: Projector, x: torch.Tensor, in_shape, out_shape, fn):
    lead = _batched(x, in_shape, "input")
    x = x.detach().to(device=proj.device, dtype=torch.float32).contiguous()
    flat = x.reshape((-1,) + tuple(in_shape))
    out = torch.empty((flat.shape[0],) + tuple(out_shape), dtype=torch.float32, device=proj.device)
    stream = torch.cuda.current_stream(proj.device)
    for i in range(flat.shape[0]):
        fn(proj.plan, flat[i], out[i], stream)
    return out.reshape(tuple(lead) + tuple(out_shape))


class _Project(torch.autograd.Function):
    @staticmethod
    def forward(ctx, vol, proj):
        ctx.proj = proj
        ctx.in_dtype, ctx.in_device = vol.dtype, vol.device
        return _apply(proj, vol, proj.vol_shape, proj.sino_shape, ctp_forward)

    @staticmethod
    def backward(ctx, grad):
        g = _Backproject.apply(grad, ctx.proj)
        return g.to(dtype=ctx.in_dtype, device=ctx.in_device), None


class _Backproject(torch.autograd.Function):
    @staticmethod
    def forward(ctx, sino, proj):
        ctx.proj = proj
        ctx.in_dtype, ctx.in_device = sino.dtype, sino.device
        return _apply(proj, sino, proj.sino_shape, proj.vol_shape, ctp_backward)

    @staticmethod
    def backward(ctx, grad):
        g = _Project.apply(grad, ctx.proj)
        return g.to(dtype=ctx.in_dtype, device=ctx.in_device), None


def _filter_fn(vw, ramp, transpose, pw):
    def fn(plan, x, out, stream):
        ctp_ramp_filter(plan, x, out, vw, ramp, transpose, stream, pw)
    return fn


class _Filter(torch.autograd.Function):
    @staticmethod
    def forward(ctx, sino, proj, vw, ramp, transpose=False, pw=None):
        ctx.proj, ctx.vw, ctx.ramp, ctx.transpose, ctx.pw = proj, vw, ramp, transpose, pw
        ctx.in_dtype, ctx.in_device = sino.dtype, sino.device
        return _apply(proj, sino, proj.sino_shape, proj.sino_shape,
                      _filter_fn(vw, ramp, transpose, pw))

    @staticmethod
    def backward(ctx, grad):
        g = _Filter.apply(grad, ctx.proj, ctx.vw, ctx.ramp, not ctx.transpose, ctx.pw)
        return g.to(dtype=ctx.in_dtype, device=ctx.in_device), None, None, None, None, None


class _Gather(torch.autograd.Function):
    @staticmethod
    def forward(ctx, sino, proj):
        ctx.proj = proj
        ctx.in_dtype, ctx.in_device = sino.dtype, sino.device
        return _apply(proj, sino, proj.sino_shape, proj.vol_shape, ctp_weighted_backproject)

    @staticmethod
    def backward(ctx, grad):
        g = _GatherT.apply(grad, ctx.proj)
        return g.to(dtype=ctx.in_dtype, device=ctx.in_device), None


class _GatherT(torch.autograd.Function):
    @staticmethod
    def forward(ctx, vol, proj):
        ctx.proj = proj
        ctx.in_dtype, ctx.in_device = vol.dtype, vol.device
        return _apply(proj, vol, proj.vol_shape, proj.sino_shape,
                      ctp_weighted_backproject_transpose)

    @staticmethod
    def backward(ctx, grad):
        g = _Gather.apply(grad, ctx.proj)
        return g.to(dtype=ctx.in_dtype, device=ctx.in_device), None


# ------------------------------------------------------------ geometry gradients
FRAME_NAMES = ("src", "det_centre", "det_u", "det_v")


def project_with_geometry(vol: torch.Tensor, geometry: Geometry, volume: Volume,
                          src: torch.Tensor, det_centre: torch.Tensor, det_u: torch.Tensor,
                          det_v: torch.Tensor, path: str = "auto",
                          pixel_offsets: torch.Tensor | None = None) -> torch.Tensor:
    """A vol with the per-view frames as differentiable inputs: the gradient
    with respect to each frame tensor (n_views, 3) is the first-order geometry
    gradient of the pages ("first-order source / centre / axis gradients";
    trajectory tensors that require gradients receive geometry gradients,
    README "Arbitrary trajectories").  ``geometry`` supplies the detector size,
    pitches and offsets; its frame arrays are replaced by the tensors' values
    (a plan is built for them on every call).  ``pixel_offsets`` (n_v, n_u, 3)
    or (n_views, n_v, n_u, 3), optional: a curved detector's per-pixel (t, s,
    e) offsets along det_u, det_v and the unit normal, shared by the views or
    one table per view, replacing ``geometry.pixel_offsets``; its
    gradient is the first-order surface gradient (README "Curved detectors":
    projection supports first-order surface gradients).  vol: (..., D, H, W);
    the geometry and surface gradients sum over leading dims.  First order."""
    return _ProjectGeometry.apply(vol, geometry, volume, path, pixel_offsets, src, det_centre,
                                  det_u, det_v)


class _ProjectGeometry(torch.autograd.Function):
    @staticmethod
    def forward(ctx, vol, geometry, volume, path, offsets, *frames):
        values = [f.detach().to(device="cpu", dtype=torch.float32).contiguous().numpy()
                  for f in frames]
        geo = dataclasses.replace(geometry, **dict(zip(FRAME_NAMES, values)))
        ctx.off_meta = None
        if offsets is not None:
            geo = dataclasses.replace(
                geo, pixel_offsets=offsets.detach().to(device="cpu", dtype=torch.float32)
                .contiguous().numpy())
            ctx.off_meta = (offsets.dtype, offsets.device, tuple(offsets.shape))
        proj = Projector(geo, volume, path)
        ctx.proj = proj
        ctx.frame_meta = [(f.dtype, f.device) for f in frames]
        ctx.in_dtype, ctx.in_device = vol.dtype, vol.device
        out = _apply(proj, vol, proj.vol_shape, proj.sino_shape, ctp_forward)
        ctx.save_for_backward(vol.detach().to(device=proj.device, dtype=torch.float32))
        return out

    @staticmethod
    def backward(ctx, grad):
        (vol,) = ctx.saved_tensors
        proj = ctx.proj
        g_vol = None
        if ctx.needs_input_grad[0]:
            g_vol = _Backproject.apply(grad, proj).to(dtype=ctx.in_dtype, device=ctx.in_device)
        g_frames = [None] * 4
        g_off = None
        want_frames = any(ctx.needs_input_grad[5:])
        want_off = ctx.off_meta is not None and ctx.needs_input_grad[4]
        if want_frames or want_off:
            grad = grad.detach().to(device=proj.device, dtype=torch.float32).contiguous()
            _batched(grad, proj.sino_shape, "grad")
            v = vol.reshape((-1,) + tuple(proj.vol_shape))
            gr = grad.reshape((-1,) + tuple(proj.sino_shape))
            stream = torch.cuda.current_stream(proj.device)
            if want_frames:
                total = torch.zeros((proj.sino_shape[0], 4, 3), dtype=torch.float64,
                                    device=proj.device)
                part = torch.empty_like(total)
                for i in range(gr.shape[0]):   # leading dims of vol and grad agree
                    ctp_geometry_vjp(proj.plan, v[i].contiguous(), gr[i].contiguous(), part,
                                     stream)
                    total += part
                for q, (dt, dev) in enumerate(ctx.frame_meta):
                    if ctx.needs_input_grad[5 + q]:
                        g_frames[q] = total[:, q, :].to(dtype=dt, device=dev)
            if want_off:
                # (n_v, n_u, 3) shared by the views, or (n_views, n_v, n_u, 3)
                total = torch.zeros(ctx.off_meta[2], dtype=torch.float64, device=proj.device)
                part = torch.empty_like(total)
                for i in range(gr.shape[0]):
                    ctp_surface_vjp(proj.plan, v[i].contiguous(), gr[i].contiguous(), part,
                                    stream)
                    total += part
                g_off = total.to(dtype=ctx.off_meta[0], device=ctx.off_meta[1])
        return (g_vol, None, None, None, g_off, *g_frames)
