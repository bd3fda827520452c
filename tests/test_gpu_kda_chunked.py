"""The KDA variant's chunked prefill on the tensor cores (gdn_kda_forward_chunked) against
the oracle's KDA recurrence and against the token-form kernel (gdn_kda_forward):

* o and S_out on ragged varlen batches (several chunks, ragged tails, one-token and empty
  sequences), both head sizes (64, 128, Dk != Dv), key heads shared by value heads
  under both head maps, a start state and in-place state;
* gates that decay fast (large a_log), where a chunk's cumulative decay underflows and
  every 16-row block's own pairs are summed channel by channel; and chunks where only
  some blocks decay that fast, so both ways of forming a block's pairs meet in one A;
* unsupported shapes are refused before anything runs.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gdn_harness import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch


def _dev(torch, a, dt=None):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda", dtype=dt or torch.float32)


def _case(Hk, Hv, Dk, Dv, seqlens, head_map=0, seed=5, a_log_shift=0.0):
    wl = W.custom(dtype="bf16", seed=seed, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, seqlens=seqlens,
                  S0_std=0.3, dt_bias_std=0.3, packed=False, head_map=head_map)
    inp = W.generate(wl)
    alpha, b_alpha = W.generate_kda_gates(wl)
    a_log = (inp.a_log + np.float32(a_log_shift)).astype(np.float32)
    return wl, inp, alpha, b_alpha, a_log


def _run_chunked(torch, gdn, wl, inp, alpha, b_alpha, a_log, in_place=False):
    td = torch.bfloat16
    T, N = wl.total_tokens, len(inp.cu_seqlens) - 1
    off, NC = gdn.gdn_plan(inp.cu_seqlens)
    q, k, v = (_dev(torch, x, td) for x in (inp.q, inp.k, inp.v))
    S_in = None if inp.S0 is None else _dev(torch, inp.S0)
    S_out = S_in if in_place else torch.full((N, wl.Hv, wl.Dk, wl.Dv), float("nan"),
                                              device="cuda")
    o = torch.full((T, wl.Hv * wl.Dv), float("nan"), device="cuda", dtype=td)
    shape = gdn.make_shape(wl.Hk, wl.Hv, wl.Dk, wl.Dv, N, NC, T, "bf16", wl.scale_value(),
                           wl.head_map)
    ws = torch.empty(max(256, gdn.gdn_kda_forward_chunked_workspace_bytes(shape)),
                     dtype=torch.uint8, device="cuda")
    gdn.gdn_kda_forward_chunked(shape, q, k, v, _dev(torch, alpha), _dev(torch, inp.beta_raw),
                                _dev(torch, a_log), _dev(torch, b_alpha),
                                _dev(torch, inp.cu_seqlens, torch.int32),
                                _dev(torch, off, torch.int32), S_in, S_out, o, ws)
    status = gdn.gdn_read_device_status(ws)
    assert status == 0, gdn.gdn_status_string(status)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), S_out.cpu().numpy()


def _run_token(torch, gdn, wl, inp, alpha, b_alpha, a_log):
    td = torch.bfloat16
    T, N = wl.total_tokens, len(inp.cu_seqlens) - 1
    q, k, v = (_dev(torch, x, td) for x in (inp.q, inp.k, inp.v))
    S_in = None if inp.S0 is None else _dev(torch, inp.S0)
    S_out = torch.full((N, wl.Hv, wl.Dk, wl.Dv), float("nan"), device="cuda")
    o = torch.full((T, wl.Hv * wl.Dv), float("nan"), device="cuda", dtype=td)
    shape = gdn.make_shape(wl.Hk, wl.Hv, wl.Dk, wl.Dv, N, 0, T, "bf16", wl.scale_value(),
                           wl.head_map)
    gdn.gdn_kda_forward(shape, q, k, v, _dev(torch, alpha), _dev(torch, inp.beta_raw),
                        _dev(torch, a_log), _dev(torch, b_alpha),
                        _dev(torch, inp.cu_seqlens, torch.int32), S_in, S_out, o)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), S_out.cpu().numpy()


def _ref(wl, inp, alpha, b_alpha, a_log):
    return oracle.kda_forward(inp.q, inp.k, inp.v, alpha, inp.beta_raw, a_log, b_alpha,
                              inp.cu_seqlens, inp.S0, Hk=wl.Hk, Hv=wl.Hv, Dk=wl.Dk, Dv=wl.Dv,
                              scale=wl.scale_value(), head_map=wl.head_map)


@pytest.mark.parametrize("Hk,Hv,Dk,Dv,seqlens,head_map", [
    (2, 6, 128, 128, (300, 1, 0, 129), 0),     # tails, one-token and empty sequences
    (1, 3, 64, 64, (200,), 0),
    (2, 4, 128, 64, (64, 127), 1),             # Dk != Dv, modulo head map
    (4, 4, 64, 128, (190, 66), 0),             # v_repeat 1
])
def test_chunked_kda_matches_the_oracle_and_the_token_form(torch_cuda, Hk, Hv, Dk, Dv, seqlens,
                                                           head_map):
    torch = torch_cuda
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, alpha, b_alpha, a_log = _case(Hk, Hv, Dk, Dv, seqlens, head_map)
    o, S = _run_chunked(torch, gdn, wl, inp, alpha, b_alpha, a_log)
    o_ref, S_ref = _ref(wl, inp, alpha, b_alpha, a_log)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    assert rel_err(o, o_ref) <= TOL["bf16"], rel_err(o, o_ref)
    assert rel_err(S, S_ref) <= TOL["bf16"], rel_err(S, S_ref)
    o_t, S_t = _run_token(torch, gdn, wl, inp, alpha, b_alpha, a_log)
    assert rel_err(o, o_t) <= TOL["bf16"] and rel_err(S, S_t) <= TOL["bf16"]


def test_fast_decaying_gates_stay_finite_and_match(torch_cuda):
    """a_log raised by 3 (decay rates ~20 times larger): the cumulative per-channel decay
    over a chunk underflows to zero; the pairwise sums never form e^{-G}."""
    torch = torch_cuda
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, alpha, b_alpha, a_log = _case(2, 4, 128, 128, (256, 90), a_log_shift=3.0, seed=9)
    o, S = _run_chunked(torch, gdn, wl, inp, alpha, b_alpha, a_log)
    o_ref, S_ref = _ref(wl, inp, alpha, b_alpha, a_log)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(S, S_ref) <= TOL["bf16"]


def test_blocks_with_fast_and_slow_gates_mix(torch_cuda):
    """alpha raised by 12 on rows 16-31 of every chunk: those blocks decay by more than
    e^60 over their 16 rows (their own pairs are summed channel by channel), the others
    go through the block products whole."""
    torch = torch_cuda
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, alpha, b_alpha, a_log = _case(2, 4, 128, 128, (200, 70, 33), seed=13)
    cu = inp.cu_seqlens
    for n in range(len(cu) - 1):
        rows = np.arange(cu[n], cu[n + 1])
        band = rows[((rows - cu[n]) % 64 >= 16) & ((rows - cu[n]) % 64 < 32)]
        alpha[band] += np.float32(12.0)
    o, S = _run_chunked(torch, gdn, wl, inp, alpha, b_alpha, a_log)
    o_ref, S_ref = _ref(wl, inp, alpha, b_alpha, a_log)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    assert rel_err(o, o_ref) <= TOL["bf16"], rel_err(o, o_ref)
    assert rel_err(S, S_ref) <= TOL["bf16"], rel_err(S, S_ref)


def test_in_place_state(torch_cuda):
    torch = torch_cuda
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, alpha, b_alpha, a_log = _case(2, 4, 128, 128, (150, 70), seed=11)
    o, S = _run_chunked(torch, gdn, wl, inp, alpha, b_alpha, a_log, in_place=True)
    o_ref, S_ref = _ref(wl, inp, alpha, b_alpha, a_log)
    assert rel_err(o, o_ref) <= TOL["bf16"] and rel_err(S, S_ref) <= TOL["bf16"]


def test_unsupported_shapes_are_refused(torch_cuda):
    torch = torch_cuda
    import gated_deltanet_backward_gb300 as gdn
    for dtype, Dk, Dv in (("f32", 128, 128), ("bf16", 32, 128), ("bf16", 128, 16)):
        shape = gdn.make_shape(1, 2, Dk, Dv, 1, 1, 10, dtype)
        assert gdn.gdn_kda_forward_chunked_workspace_bytes(shape) == 0


@pytest.mark.slow
def test_27b_head_shape_against_the_oracle(torch_cuda):
    """16 key heads shared by 48 value heads of 128, one 1024-token sequence with a start
    state: every value head against the oracle, and against the token form."""
    torch = torch_cuda
    import gated_deltanet_backward_gb300 as gdn
    wl, inp, alpha, b_alpha, a_log = _case(16, 48, 128, 128, (1024,), seed=21)
    o, S = _run_chunked(torch, gdn, wl, inp, alpha, b_alpha, a_log)
    o_ref, S_ref = _ref(wl, inp, alpha, b_alpha, a_log)
    assert rel_err(o, o_ref) <= TOL["bf16"], rel_err(o, o_ref)
    assert rel_err(S, S_ref) <= TOL["bf16"], rel_err(S, S_ref)
    o_t, S_t = _run_token(torch, gdn, wl, inp, alpha, b_alpha, a_log)
    assert rel_err(o, o_t) <= TOL["bf16"] and rel_err(S, S_t) <= TOL["bf16"]
