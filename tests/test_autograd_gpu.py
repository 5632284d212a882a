"""Differentiable wrapper: gradients are the matched operators, batch dims loop,
second derivatives work (data Hessian-vector products)."""

import numpy as np
import pytest

from cases import ci, geometry_of, rel_l2, volume_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def proj():
    import torch  # noqa: F401
    from back_projection_ctp_b300.autograd import Projector
    w = ci.small_cases()[3]
    return Projector(geometry_of(w, ci.frames(w)), volume_of(w))


def test_gradient_of_projection_is_backprojection(proj):
    import torch
    x = torch.randn(proj.vol_shape, device="cuda", requires_grad=True)
    g = torch.randn(proj.sino_shape, device="cuda")
    (proj.project(x) * g).sum().backward()
    ref = proj.backproject(g)
    assert rel_l2(x.grad.cpu().numpy(), ref.cpu().numpy()) <= 1e-6


def test_gradient_of_backprojection_is_projection(proj):
    import torch
    y = torch.randn(proj.sino_shape, device="cuda", requires_grad=True)
    h = torch.randn(proj.vol_shape, device="cuda")
    (proj.backproject(y) * h).sum().backward()
    ref = proj.project(h)
    assert rel_l2(y.grad.cpu().numpy(), ref.cpu().numpy()) <= 1e-6


def test_batch_and_channel_dims_and_empty_batch(proj):
    import torch
    x = torch.randn((2, 3) + proj.vol_shape, device="cuda")
    p = proj.project(x)
    assert p.shape == (2, 3) + proj.sino_shape
    for i in range(2):
        for j in range(3):
            assert torch.equal(p[i, j], proj.project(x[i, j]))
    e = proj.project(torch.zeros((0,) + proj.vol_shape, device="cuda"))
    assert e.shape == (0,) + proj.sino_shape
    with pytest.raises(ValueError):
        proj.project(torch.zeros((4, 5, 6), device="cuda"))


def test_hessian_vector_product_of_least_squares(proj):
    """loss = 0.5 ||A x - b||^2: grad = A^T (A x - b), Hessian-vector product = A^T A v."""
    import torch
    x = torch.randn(proj.vol_shape, device="cuda", requires_grad=True)
    b = torch.randn(proj.sino_shape, device="cuda")
    v = torch.randn(proj.vol_shape, device="cuda")
    loss = 0.5 * ((proj.project(x) - b) ** 2).sum()
    (grad,) = torch.autograd.grad(loss, x, create_graph=True)
    (hv,) = torch.autograd.grad((grad * v).sum(), x)
    ref = proj.backproject(proj.project(v))
    assert rel_l2(hv.cpu().numpy(), ref.cpu().numpy()) <= 1e-5
    ref_g = proj.backproject(proj.project(x.detach()) - b)
    assert rel_l2(grad.detach().cpu().numpy(), ref_g.cpu().numpy()) <= 1e-5


def test_double_precision_inputs_keep_their_dtype_for_gradients(proj):
    import torch
    x = torch.randn(proj.vol_shape, device="cuda", dtype=torch.float64, requires_grad=True)
    proj.project(x).sum().backward()
    assert x.grad.dtype == torch.float64


def test_fdk_gradient_is_the_transposed_pipeline(proj, oracle_mod):
    """d<FDK(y), h>/dy = F^T B^T h, checked against the float64 oracle's transposes."""
    import torch
    from oracle import fdk as ofdk
    import back_projection_ctp_b300 as ctp
    w = ci.small_cases()[3]
    scan = oracle_mod.Scan.from_workload(w, ci.frames(w))
    vw_h = ctp.full_scan_view_weights(w.n_views)
    vw = torch.from_numpy(vw_h).cuda()
    y = torch.randn(proj.sino_shape, device="cuda", requires_grad=True)
    h = torch.randn(proj.vol_shape, device="cuda")
    out = proj.fdk(y, vw)
    ref_fwd = ofdk.fdk(scan, y.detach().cpu().numpy(), vw_h)
    assert rel_l2(out.detach().cpu().numpy(), ref_fwd) <= 1e-5
    (out * h).sum().backward()
    hh = h.cpu().numpy().astype(np.float64)
    ref = ofdk.filter_sinogram_transpose(scan, ofdk.weighted_backproject_transpose(scan, hh), vw_h)
    assert rel_l2(y.grad.cpu().numpy(), ref) <= 1e-4


def test_fdk_batch_dims(proj):
    import torch
    y = torch.randn((2,) + proj.sino_shape, device="cuda")
    out = proj.fdk(y)
    assert out.shape == (2,) + proj.vol_shape
    one = proj.fdk(y[1])
    assert rel_l2(out[1].cpu().numpy(), one.cpu().numpy()) == 0.0


@pytest.mark.parametrize("beam_idx", [3, 2])
def test_geometry_gradients_through_autograd(oracle_mod, beam_idx):
    """loss = <A(frames) x, w>: the frames' .grad equals the oracle's geometry
    gradient (kink and face-plane rays carry zero weight) and x.grad = A^T w."""
    import torch
    from back_projection_ctp_b300.autograd import project_with_geometry
    w_ = ci.small_cases()[beam_idx]
    f = ci.frames(w_)
    scan = oracle_mod.Scan.from_workload(w_, f)
    skip = oracle_mod.ambiguous(scan) | oracle_mod.kinks(scan)
    wt = np.where(skip, 0.0, np.random.default_rng(5).standard_normal(scan.sino_shape))
    wt = wt.astype(np.float32)
    vol = ci.phantom(w_)
    x = torch.from_numpy(vol).cuda().requires_grad_()
    frames = [torch.from_numpy(f[k].astype(np.float64)).requires_grad_()
              for k in ("src", "det_centre", "det_u", "det_v")]
    out = project_with_geometry(x, geometry_of(w_, f), volume_of(w_), *frames)
    (out * torch.from_numpy(wt).cuda()).sum().backward()
    got = np.stack([fr.grad.numpy() for fr in frames], axis=1)
    ref = oracle_mod.geometry_vjp(scan, vol, wt.ravel())
    assert rel_l2(got, ref) <= 1e-4
    assert frames[0].grad.dtype == torch.float64
    back = oracle_mod.backward(scan, wt.ravel())
    assert rel_l2(x.grad.cpu().numpy(), back) <= 1e-4


def test_surface_gradients_through_autograd(oracle_mod):
    """loss = <A(frames, offsets) x, w> on a curved (cylindrical) detector: the
    offsets' .grad equals the oracle's surface gradient and the frames' .grad
    its curved geometry gradient (kink and face-plane rays carry zero weight)."""
    import torch
    import back_projection_ctp_b300 as ctp
    from back_projection_ctp_b300.autograd import project_with_geometry
    from test_oracle_curved_pins import _cylinder_offsets
    w_ = ci.small_cases()[3]
    f = ci.frames(ci.scaled(w_, 1.0, views=8, ragged=0))
    n_u, n_v = 29, 23
    off = _cylinder_offsets(n_u, n_v, 1000.0, 0.0131, 13.1)
    scan = oracle_mod.Scan("divergent", f["src"], f["det_centre"], f["det_u"], f["det_v"], n_u,
                           n_v, 1.0, 1.0, w_.shape, w_.spacing, w_.origin, 0.0, 0.0, 3, off)
    skip = oracle_mod.ambiguous(scan) | oracle_mod.kinks(scan)
    wt = np.where(skip, 0.0, np.random.default_rng(6).standard_normal(scan.sino_shape))
    wt = wt.astype(np.float32)
    vol = ci.phantom(w_)
    geom = ctp.Geometry(ndim=3, beam="divergent", n_u=n_u, n_v=n_v, pitch_u=1.0, pitch_v=1.0,
                        pixel_offsets=off, **f)
    x = torch.from_numpy(vol).cuda()
    offsets = torch.from_numpy(off.astype(np.float64)).requires_grad_()
    frames = [torch.from_numpy(f[k].astype(np.float64)).requires_grad_()
              for k in ("src", "det_centre", "det_u", "det_v")]
    out = project_with_geometry(x, geom, volume_of(w_), *frames, pixel_offsets=offsets)
    (out * torch.from_numpy(wt).cuda()).sum().backward()
    assert rel_l2(offsets.grad.numpy(), oracle_mod.surface_vjp(scan, vol, wt.ravel())) <= 1e-4
    got = np.stack([fr.grad.numpy() for fr in frames], axis=1)
    assert rel_l2(got, oracle_mod.geometry_vjp(scan, vol, wt.ravel())) <= 1e-4
