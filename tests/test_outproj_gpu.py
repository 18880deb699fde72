"""The norm fused into the out_proj GEMM (ggrn_norm_outproj), on the GPU.

Two parts are checked against the oracle, each at the precision it has:

* the A operand the GEMM used (written to ``a_out``): the Mamba-2 norm of the
  "gated_group_rmsnorm" page's math block, under the same rules as the norm
  kernels (tests/tolerance.py: equal to the oracle's output except explained
  flips of the intermediate cast);
* Z = A W_out^T in bf16 with f32 sums, against the oracle's A times W_out in
  f64.  Per output element the stated tolerance is
      ulp_bf16(|Z_ref|)                        the final rounding (and slack)
    + 4 u K sqrt(mean_k (a_k w_nk)^2)           f32 sums over K terms, u = 2^-24
                                                (about ten times the spread of a
                                                K-term running sum's error)
    + sum_{k may flip} 2 ulp(a_k) |w_nk|        A elements whose intermediate
                                                may flip (tolerance.mamba2_flip_mask)
  with K = width.  Every row of A and a sample of rows of Z are compared.
"""
import pytest
import torch

import ggrn_inputs
import gated_group_rmsnorm_gb300 as g
import oracle
from tests import gpu_util
from tests.tolerance import U, assert_parity, mamba2_flip_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.load()


def _ulp_bf16(x: torch.Tensor) -> torch.Tensor:
    e = torch.floor(torch.log2(x.abs().clamp(min=2.0 ** -126)))
    return torch.pow(2.0, e - 7)


def _z_check(z_got, host, w_out, rows_idx, wl):
    """Z rows `rows_idx` against the oracle's A times W_out (f64), under the
    tolerance of the module docstring; returns (max error / tolerance, n)."""
    y = host.y[rows_idx]
    gate = host.gate[rows_idx]
    a, t, pre = oracle.default().forward_detail(y.contiguous(), gate.contiguous(), host.w,
                                                group_size=wl.group_size, eps=wl.eps, mode=0)
    a64 = a.double()
    w64 = w_out.double()
    z_ref = a64 @ w64.T
    K = a.shape[1]
    sigma = torch.sqrt(((a64 ** 2) @ (w64 ** 2).T) / K)
    near = mamba2_flip_mask(t, pre, gate.contiguous(), wl.group_size)
    flip = ((2 * _ulp_bf16(a64)) * near.double()) @ w64.abs().T
    tol = _ulp_bf16(z_ref) + 4 * U * K * sigma + flip
    err = (z_got.double() - z_ref).abs()
    assert bool(torch.isfinite(z_got.double()).all())
    ratio = float((err / tol).max())
    assert bool((err <= tol).all()), (ratio, float(err.max()))
    return ratio, err.numel()


def _run(wl, d_model, rows_sample, packed=False, seed=0):
    host = ggrn_inputs.make_inputs(wl, seed=seed)
    if packed:
        # y and gate as column ranges of one packed buffer (the fused in-proj layout)
        buf = torch.zeros((wl.rows, 2 * wl.width + 64), dtype=wl.dtype)
        buf[:, :wl.width] = host.y
        buf[:, wl.width:2 * wl.width] = host.gate
        host = ggrn_inputs.Inputs(y=buf[:, :wl.width], gate=buf[:, wl.width:2 * wl.width],
                                  w=host.w, packed=buf)
    dev = gpu_util.to_device(host)
    w_out = ggrn_inputs.make_outproj_weight(d_model, wl.width, seed=seed + 1)
    a_out = torch.empty((wl.rows, wl.width), dtype=torch.bfloat16, device="cuda")
    g.fault_status(clear=True)
    z = g.norm_outproj(dev.y, dev.gate, dev.w, w_out.cuda(), group_size=wl.group_size,
                       eps=wl.eps, a_out=a_out)
    z2 = g.norm_outproj(dev.y, dev.gate, dev.w, w_out.cuda(), group_size=wl.group_size,
                        eps=wl.eps)
    torch.cuda.synchronize()
    assert g.fault_status() == 0
    assert torch.equal(z.view(torch.int16), z2.view(torch.int16)), "a_out changed z or runs differ"
    res = gpu_util.compare_all_rows(a_out.cpu(), host, wl.group_size, wl.eps, 0)
    assert_parity(res, "A operand")
    idx = torch.tensor(rows_sample)
    ratio, n = _z_check(z.cpu()[idx], host, w_out, idx, wl)
    print(f"norm_outproj {wl.rows}x{wl.width}x{d_model}: A {res}; Z {n} outputs, "
          f"max error {ratio:.3f} of the tolerance")
    return z


def test_small_shapes():
    # one tile per row block (no cluster), two (a pair of CTAs shares each A
    # block) and four or more (clusters of four)
    for rows, width, gs, d_model in ((128, 256, 64, 64), (256, 1024, 256, 512),
                                     (384, 960 * 2, 960, 480), (128, 640, 128, 96),
                                     (256, 1024, 256, 1024), (128, 1920, 960, 1920),
                                     (256, 512, 64, 4096)):
        wl = ggrn_inputs.Workload("op", rows, width, gs, torch.bfloat16, 0, 1e-5, sat_frac=0.01)
        _run(wl, d_model, list(range(rows)))


def test_packed_inproj_views():
    wl = ggrn_inputs.Workload("op", 256, 1920, 960, torch.bfloat16, 0, 1e-5)
    _run(wl, 480, list(range(0, 256, 3)), packed=True, seed=5)


@pytest.mark.parametrize("d_model", [3840, 7680])
def test_prefill_shape(d_model):
    """The Mamba-2 prefill shape (4096 x 7680, groups of 960) into an out_proj
    of d_model outputs; every row of A, 48 rows of Z (all columns)."""
    wl = ggrn_inputs.WORKLOADS["mamba2_prefill"]
    gen = torch.Generator().manual_seed(d_model)
    rows = sorted(set([0, 127, 128, wl.rows - 1] + torch.randint(0, wl.rows, (44,),
                                                                 generator=gen).tolist()))
    _run(wl, d_model, rows)


def test_unsupported_shapes_are_refused():
    y = torch.zeros((100, 128), dtype=torch.bfloat16, device="cuda")  # rows not a multiple of 128
    w = torch.ones(128, device="cuda")
    wo = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GgrnError) as ei:
        g.norm_outproj(y, y.clone(), w, wo, group_size=64, eps=1e-5)
    assert ei.value.status == 7
    y = torch.zeros((128, 100), dtype=torch.bfloat16, device="cuda")  # width not a multiple of 64
    with pytest.raises(g.GgrnError) as ei:
        g.norm_outproj(y, y.clone(), torch.ones(100, device="cuda"),
                       torch.zeros((64, 100), dtype=torch.bfloat16, device="cuda"),
                       group_size=100, eps=1e-5)
    assert ei.value.status == 7
