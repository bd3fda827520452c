"""The layer steps on either side of the recurrence (causal depthwise conv1d + SiLU, gated
RMSNorm) on the GPU against the oracle, element by element, forward and backward:

* ragged varlen batches (empty sequences, sequences shorter than the kernel, several
  token tiles and a ragged tail), channel counts that leave a partial block, strided
  row views, every kernel size 1..4 and every head size;
* the full 27B-shaped layer (4096 tokens, 10240 packed channels, 48 value heads of 128)
  against the oracle on every element;
* the weight gradients bit-identical run to run; zero tokens; rejected arguments;
* the composition conv -> recurrence -> norm and back through the C ABI, against the
  oracle's composition.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gdn_harness import TOL, rel_err

pytestmark = pytest.mark.gpu


def _torch():
    return pytest.importorskip("torch")


def _dev(torch, a, dt=None):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda", dtype=dt or torch.float32)


def _td(torch, dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def _conv_case(dtype, Hk, Hv, D, seqlens, K, w_range=0.7, seed=0):
    wl = W.custom(dtype=dtype, seed=seed, Hk=Hk, Hv=Hv, Dk=D, Dv=D, seqlens=seqlens)
    return W.generate_layer_steps(wl, K=K, w_range=w_range)


def _run_conv(torch, gdn, inp, dtype, pad=0, want_dw=True):
    """GPU conv forward and backward; `pad` extra columns make x, y, dy, dx strided views."""
    td = _td(torch, dtype)
    T, C = inp.x.shape

    def view(a):
        buf = torch.zeros((T, C + pad), device="cuda", dtype=td)
        buf[:, :C] = _dev(torch, a, td)
        return buf[:, :C]

    x, dy = view(inp.x), view(inp.dy_conv)
    y = torch.full((T, C + pad), float("nan"), device="cuda", dtype=td)[:, :C]
    dx = torch.full((T, C + pad), float("nan"), device="cuda", dtype=td)[:, :C]
    w = _dev(torch, inp.w)
    cu = _dev(torch, inp.cu_seqlens, torch.int32)
    gdn.gdn_conv1d_silu_forward(x, w, cu, y)
    dw = ws = None
    if want_dw:
        dw = torch.full_like(w, float("nan"))
        ws = torch.empty(max(16, gdn.gdn_conv1d_silu_workspace_bytes(T, C, w.shape[1])),
                         dtype=torch.uint8, device="cuda")
    gdn.gdn_conv1d_silu_backward(x, w, cu, dy, dx, dw, ws)
    torch.cuda.synchronize()
    return (y.float().cpu().numpy(), dx.float().cpu().numpy(),
            None if dw is None else dw.cpu().numpy())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_conv_matches_the_oracle_on_ragged_batches(dtype, K):
    torch = _torch()
    import gated_deltanet_backward_gb300 as gdn
    # 2 Hk D + Hv D = 2*1*32 + 3*32 = 160 channels: a partial block of channel vectors;
    # 600 tokens: three token tiles, the last ragged; empty and 1-, 2-, 3-token sequences
    inp = _conv_case(dtype, 1, 3, 32, (2, 0, 1, 300, 3, 0, 250, 44), K, seed=K)
    y, dx, dw = _run_conv(torch, gdn, inp, dtype)
    y_ref = oracle.conv1d_silu_forward(inp.x, inp.w, inp.cu_seqlens)
    dx_ref, dw_ref = oracle.conv1d_silu_backward(inp.x, inp.w, inp.cu_seqlens, inp.dy_conv)
    assert rel_err(y, y_ref) <= TOL[dtype]
    assert rel_err(dx, dx_ref) <= TOL[dtype]
    assert rel_err(dw, dw_ref) <= TOL["f32"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_on_strided_views_and_without_dw(dtype):
    torch = _torch()
    import gated_deltanet_backward_gb300 as gdn
    inp = _conv_case(dtype, 2, 4, 16, (37, 290), 4, seed=3)
    y, dx, dw = _run_conv(torch, gdn, inp, dtype, pad=24, want_dw=False)
    assert dw is None
    assert rel_err(y, oracle.conv1d_silu_forward(inp.x, inp.w, inp.cu_seqlens)) <= TOL[dtype]
    dx_ref, _ = oracle.conv1d_silu_backward(inp.x, inp.w, inp.cu_seqlens, inp.dy_conv)
    assert rel_err(dx, dx_ref) <= TOL[dtype]


def test_conv_dw_is_bit_reproducible():
    torch = _torch()
    import gated_deltanet_backward_gb300 as gdn
    inp = _conv_case("bf16", 2, 6, 64, (700, 333), 4, seed=9)
    _, dx1, dw1 = _run_conv(torch, gdn, inp, "bf16")
    _, dx2, dw2 = _run_conv(torch, gdn, inp, "bf16")
    assert np.array_equal(dw1, dw2) and np.array_equal(dx1, dx2)


def _run_norm(torch, gdn, inp, dtype, H, eps, pad=0, want_dg=True):
    td = _td(torch, dtype)
    T, Wd = inp.o.shape

    def view(a):
        buf = torch.zeros((T, Wd + pad), device="cuda", dtype=td)
        buf[:, :Wd] = _dev(torch, a, td)
        return buf[:, :Wd]

    def out():
        return torch.full((T, Wd + pad), float("nan"), device="cuda", dtype=td)[:, :Wd]

    o, z, dy = view(inp.o), view(inp.z), view(inp.dy_norm)
    y, d_o, dz = out(), out(), out()
    gamma = _dev(torch, inp.gamma)
    gdn.gdn_gated_rmsnorm_forward(o, z, gamma, y, eps)
    dg = ws = None
    if want_dg:
        dg = torch.full_like(gamma, float("nan"))
        ws = torch.empty(gdn.gdn_gated_rmsnorm_workspace_bytes(gamma.numel()), dtype=torch.uint8,
                         device="cuda")
    gdn.gdn_gated_rmsnorm_backward(o, z, gamma, dy, d_o, dz, eps, dg, ws)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().numpy()
    return f(y), f(d_o), f(dz), None if dg is None else dg.cpu().numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("D,H,eps", [(16, 3, 1e-6), (32, 1, 0.25), (64, 5, 1e-5), (128, 2, 1e-6)])
def test_norm_matches_the_oracle(dtype, D, H, eps):
    torch = _torch()
    import gated_deltanet_backward_gb300 as gdn
    inp = _conv_case(dtype, 1, H, D, (0, 333, 1), 4, seed=D + H)
    y, d_o, dz, dg = _run_norm(torch, gdn, inp, dtype, H, eps, pad=8 if D == 64 else 0)
    y_ref = oracle.gated_rmsnorm_forward(inp.o, inp.z, inp.gamma, H, D, eps)
    do_ref, dz_ref, dg_ref = oracle.gated_rmsnorm_backward(inp.o, inp.z, inp.gamma, inp.dy_norm,
                                                            H, D, eps)
    assert rel_err(y, y_ref) <= TOL[dtype]
    assert rel_err(d_o, do_ref) <= TOL[dtype]
    assert rel_err(dz, dz_ref) <= TOL[dtype]
    assert rel_err(dg, dg_ref) <= TOL["f32"]


def test_norm_dgamma_is_bit_reproducible():
    torch = _torch()
    import gated_deltanet_backward_gb300 as gdn
    inp = _conv_case("bf16", 2, 8, 128, (1000, 200), 4, seed=4)
    r1 = _run_norm(torch, gdn, inp, "bf16", 8, 1e-6)
    r2 = _run_norm(torch, gdn, inp, "bf16", 8, 1e-6)
    for a, b in zip(r1, r2):
        assert np.array_equal(a, b)


@pytest.mark.slow
def test_full_layer_against_the_oracle_on_every_element():
    """The 27B-shaped layer: 4096 tokens, 10240 packed channels, 48 heads of 128, bf16."""
    torch = _torch()
    import gated_deltanet_backward_gb300 as gdn
    wl = W.get("l27b_bf16")
    inp = W.generate_layer_steps(wl)
    y, dx, dw = _run_conv(torch, gdn, inp, "bf16")
    assert rel_err(y, oracle.conv1d_silu_forward(inp.x, inp.w, inp.cu_seqlens)) <= TOL["bf16"]
    dx_ref, dw_ref = oracle.conv1d_silu_backward(inp.x, inp.w, inp.cu_seqlens, inp.dy_conv)
    assert rel_err(dx, dx_ref) <= TOL["bf16"]
    assert rel_err(dw, dw_ref) <= TOL["f32"]
    H, D = wl.Hv, wl.Dv
    y, d_o, dz, dg = _run_norm(torch, gdn, inp, "bf16", H, 1e-6)
    assert rel_err(y, oracle.gated_rmsnorm_forward(inp.o, inp.z, inp.gamma, H, D, 1e-6)) \
        <= TOL["bf16"]
    do_ref, dz_ref, dg_ref = oracle.gated_rmsnorm_backward(inp.o, inp.z, inp.gamma, inp.dy_norm,
                                                            H, D, 1e-6)
    assert rel_err(d_o, do_ref) <= TOL["bf16"]
    assert rel_err(dz, dz_ref) <= TOL["bf16"]
    assert rel_err(dg, dg_ref) <= TOL["f32"]


def test_zero_tokens_write_zero_weight_gradients():
    torch = _torch()
    import gated_deltanet_backward_gb300 as gdn
    z2 = lambda c: torch.zeros((0, c), device="cuda")
    w = torch.ones((16, 3), device="cuda")
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    dw = torch.full_like(w, float("nan"))
    gdn.gdn_conv1d_silu_forward(z2(16), w, cu, z2(16))
    gdn.gdn_conv1d_silu_backward(z2(16), w, cu, z2(16), z2(16), dw,
                                 torch.empty(256, dtype=torch.uint8, device="cuda"))
    g = torch.ones(32, device="cuda")
    dg = torch.full_like(g, float("nan"))
    gdn.gdn_gated_rmsnorm_backward(z2(64), z2(64), g, z2(64), z2(64), z2(64), 1e-6, dg,
                                   torch.empty(gdn.gdn_gated_rmsnorm_workspace_bytes(32),
                                               dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert (dw == 0).all() and (dg == 0).all()


def test_rejects_bad_arguments_before_launching():
    torch = _torch()
    import gated_deltanet_backward_gb300 as gdn
    T = 10
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    x = torch.zeros((T, 24), device="cuda")
    y = torch.zeros((T, 24), device="cuda")
    with pytest.raises(gdn.GdnError):                  # kernel size 5
        gdn.gdn_conv1d_silu_forward(x, torch.zeros((24, 5), device="cuda"), cu, y)
    with pytest.raises(gdn.GdnError):                  # 12 channels: not a multiple of 8
        gdn.gdn_conv1d_silu_forward(x[:, :12], torch.zeros((12, 4), device="cuda"), cu,
                                    y[:, :12])
    with pytest.raises(gdn.GdnError):                  # output overlaps the input
        gdn.gdn_conv1d_silu_forward(x, torch.zeros((24, 4), device="cuda"), cu, x)
    with pytest.raises(gdn.GdnError):                  # dw without a workspace
        gdn.gdn_conv1d_silu_backward(x, torch.zeros((24, 4), device="cuda"), cu, x, y,
                                     torch.zeros((24, 4), device="cuda"), None)
    o = torch.zeros((T, 96), device="cuda")
    with pytest.raises(gdn.GdnError):                  # head size 48
        gdn.gdn_gated_rmsnorm_forward(o, o.clone(), torch.ones(48, device="cuda"),
                                      torch.zeros_like(o), 1e-6)
    with pytest.raises(gdn.GdnError):                  # negative eps
        gdn.gdn_gated_rmsnorm_forward(o, o.clone(), torch.ones(32, device="cuda"),
                                      torch.zeros_like(o), -1.0)


def test_conv_recurrence_norm_composition_against_the_oracle():
    """x -> conv1d + SiLU -> (q | k | v) -> recurrence -> o -> gated RMSNorm -> y, and the
    gradients back to dx and dw, all through the C ABI, against the oracle's composition."""
    torch = _torch()
    import gated_deltanet_backward_gb300 as gdn
    Hk, Hv, D, K, eps = 2, 4, 32, 4, 1e-6
    wl = W.custom(dtype="f32", seed=31, Hk=Hk, Hv=Hv, Dk=D, Dv=D, seqlens=(70, 5, 130),
                  S0_std=0.2, dt_bias_std=0.2, packed=True)
    rec = W.generate(wl)
    ls = W.generate_layer_steps(wl, K=K, w_range=0.7)
    T, C = ls.x.shape
    cu_h = ls.cu_seqlens
    # oracle
    c = oracle.conv1d_silu_forward(ls.x, ls.w, cu_h)
    q, k, v = c[:, :Hk * D], c[:, Hk * D:2 * Hk * D], c[:, 2 * Hk * D:]
    kw = dict(Hk=Hk, Hv=Hv, Dk=D, Dv=D, scale=wl.scale_value())
    o_ref, _ = oracle.forward(q, k, v, rec.alpha, rec.beta_raw, rec.a_log, rec.dt_bias, cu_h,
                              rec.S0, **kw)
    y_ref = oracle.gated_rmsnorm_forward(o_ref, ls.z, ls.gamma, Hv, D, eps)
    do_ref, dz_ref, dg_ref = oracle.gated_rmsnorm_backward(o_ref, ls.z, ls.gamma, ls.dy_norm,
                                                            Hv, D, eps)
    g = oracle.backward(q, k, v, rec.alpha, rec.beta_raw, rec.a_log, rec.dt_bias, cu_h, do_ref,
                        rec.S0, None, **kw)
    dc = np.concatenate([g["dq"], g["dk"], g["dv"]], axis=1)
    dx_ref, dw_ref = oracle.conv1d_silu_backward(ls.x, ls.w, cu_h, dc)
    # GPU
    layer = gdn.Layer.create(Hk, Hv, D, D, cu_h, "f32", wl.scale_value())
    x, w, z, gamma = (_dev(torch, a) for a in (ls.x, ls.w, ls.z, ls.gamma))
    cy = torch.empty((T, C), device="cuda")
    gdn.gdn_conv1d_silu_forward(x, w, layer.cu_seqlens, cy)
    qg, kg, vg = cy[:, :Hk * D], cy[:, Hk * D:2 * Hk * D], cy[:, 2 * Hk * D:]
    alpha, beta_raw, a_log, dt_bias, S0 = (_dev(torch, a) for a in
                                           (rec.alpha, rec.beta_raw, rec.a_log, rec.dt_bias,
                                            rec.S0))
    o = torch.empty((T, Hv * D), device="cuda")
    S_T = torch.empty((len(cu_h) - 1, Hv, D, D), device="cuda")
    layer.forward(qg, kg, vg, alpha, beta_raw, a_log, dt_bias, S0, o, S_T, train=True)
    y = torch.empty_like(o)
    gdn.gdn_gated_rmsnorm_forward(o, z, gamma, y, eps)
    d_o, dz = torch.empty_like(o), torch.empty_like(o)
    dg = torch.empty_like(gamma)
    gdn.gdn_gated_rmsnorm_backward(o, z, gamma, _dev(torch, ls.dy_norm), d_o, dz, eps, dg,
                                   torch.empty(gdn.gdn_gated_rmsnorm_workspace_bytes(D),
                                               dtype=torch.uint8, device="cuda"))
    dcy = torch.empty((T, C), device="cuda")   # dq | dk | dv packed as the conv's dy
    dq, dk, dv = dcy[:, :Hk * D], dcy[:, Hk * D:2 * Hk * D], dcy[:, 2 * Hk * D:]
    dalpha, dbeta = torch.empty_like(alpha), torch.empty_like(beta_raw)
    da_log, ddt = torch.empty_like(a_log), torch.empty_like(dt_bias)
    dS0 = torch.empty_like(S0)
    layer.backward(qg, kg, vg, alpha, beta_raw, a_log, dt_bias, S0, d_o, None, dq, dk, dv,
                   dalpha, dbeta, da_log, ddt, dS0, train=True)
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    gdn.gdn_conv1d_silu_backward(x, w, layer.cu_seqlens, dcy, dx, dw,
                                 torch.empty(gdn.gdn_conv1d_silu_workspace_bytes(T, C, K),
                                             dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    f = lambda t: t.cpu().numpy()
    assert rel_err(f(y), y_ref) <= TOL["f32"]
    assert rel_err(f(dz), dz_ref) <= TOL["f32"]
    assert rel_err(f(dg), dg_ref) <= TOL["f32"]
    assert rel_err(f(dx), dx_ref) <= TOL["f32"]
    assert rel_err(f(dw), dw_ref) <= TOL["f32"]
