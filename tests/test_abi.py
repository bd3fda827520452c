"""The C-ABI library on the host (no GPU needed): it builds, loads, exports every
entry point declared in include/gdn.h, links into a plain C program, and rejects bad
arguments before any launch.  No call here reaches a kernel."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gdn():
    import __graft_entry__
    __graft_entry__._builder().build()
    import gated_deltanet_backward_gb300 as g
    return g


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(gdn_\w+)\s*\(", text, flags=re.M))
    return names


def test_every_declared_symbol_is_exported(gdn):
    declared = _declared()
    assert {"gdn_plan", "gdn_forward", "gdn_backward", "gdn_workspace_bytes",
            "gdn_saved_state_bytes", "gdn_read_device_status", "gdn_status_string"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (gdn_\w+)$", out, flags=re.M))
    assert declared <= exported, declared - exported
    lib = ctypes.CDLL(gdn.LIB_PATH)
    for name in declared:
        assert getattr(lib, name) is not None


def test_plan(gdn):
    off, nc = gdn.gdn_plan([0, 64, 64, 200, 201])
    assert list(off) == [0, 1, 1, 4, 5] and nc == 5
    off, nc = gdn.gdn_plan([0])
    assert list(off) == [0] and nc == 0
    with pytest.raises(gdn.GdnError):
        gdn.gdn_plan([0, 10, 5])
    with pytest.raises(gdn.GdnError):
        gdn.gdn_plan([3, 10])


def test_sizes(gdn):
    s = gdn.make_shape(16, 48, 128, 128, 1, 64, 4096, "bf16")
    # the fp32 chunk-start states [total_chunks, Hv, Dk, Dv] for both input dtypes
    assert gdn.gdn_saved_state_bytes(s) == 64 * 48 * 128 * 128 * 4
    assert gdn.gdn_saved_state_bytes(gdn.make_shape(2, 4, 16, 32, 1, 3, 150, "bf16")) == \
        3 * 4 * 16 * 32 * 4
    assert gdn.gdn_saved_state_bytes(gdn.make_shape(2, 4, 16, 32, 1, 3, 150, "f32")) == \
        3 * 4 * 16 * 32 * 4
    # the bf16 tiles of GDN_FLAG_BF16_SAVED_STATES (Dk, Dv >= 64) fit in the same buffer
    for Dk in (64, 128):
        for Dv in (64, 128):
            tile = -(-Dk // 64) * max(Dv, 64) * 128
            assert tile <= Dk * Dv * 4, (Dk, Dv)
    f, b = gdn.gdn_workspace_bytes(s, False), gdn.gdn_workspace_bytes(s, True)
    assert 256 < f < b and f % 256 == 0 and b % 256 == 0
    bad = gdn.make_shape(16, 48, 96, 128, 1, 64, 4096, "bf16")
    assert gdn.gdn_workspace_bytes(bad, False) == 0
    assert gdn.gdn_workspace_bytes(gdn.make_shape(16, 40, 128, 128, 1, 64, 4096, "bf16"), 1) == 0


def _fwd_args(gdn, shape, **over):
    """Fake, never-dereferenced device addresses: every call below fails a host check."""
    A = 1 << 20
    a = dict(q=A, q_ld=shape.Hk * shape.Dk * 2 + shape.Hv * shape.Dv, k=A, k_ld=None, v=A,
             v_ld=None, alpha=A, alpha_ld=shape.Hv, beta=A, beta_ld=shape.Hv, a_log=A, dt=A,
             cu=A, coff=A, S0=None, o=A, o_ld=shape.Hv * shape.Dv, S_T=None, saved=A, ws=A,
             ws_bytes=0, flags=0, stream=None)
    a["k_ld"] = a["q_ld"]
    a["v_ld"] = a["q_ld"]
    a.update(over)
    return [ctypes.byref(shape), a["q"], a["q_ld"], a["k"], a["k_ld"], a["v"], a["v_ld"],
            a["alpha"], a["alpha_ld"], a["beta"], a["beta_ld"], a["a_log"], a["dt"], a["cu"],
            a["coff"], a["S0"], a["o"], a["o_ld"], a["S_T"], a["saved"], a["ws"], a["ws_bytes"],
            a["flags"], a["stream"]]


def _device_visible():
    import torch
    return torch.cuda.is_available()


@pytest.mark.skipif(_device_visible(), reason="fake device addresses: host-only machines")
def test_forward_rejects_bad_arguments_before_launching(gdn):
    lib = gdn._lib
    s = gdn.make_shape(2, 6, 64, 64, 1, 2, 100, "f32")
    ws = gdn.gdn_workspace_bytes(s, False)
    # null q
    assert lib.gdn_forward(*_fwd_args(gdn, s, q=None, ws_bytes=ws)) == -1
    # misaligned q base and q row stride that is not a multiple of 16 bytes
    assert lib.gdn_forward(*_fwd_args(gdn, s, q=(1 << 20) + 4, ws_bytes=ws)) == -3
    assert lib.gdn_forward(*_fwd_args(gdn, s, q_ld=2 * 64 * 2 + 6 * 64 + 1, ws_bytes=ws)) == -3
    # row stride narrower than the heads it must hold
    assert lib.gdn_forward(*_fwd_args(gdn, s, q_ld=64, ws_bytes=ws)) == -1
    # workspace too small or misaligned
    assert lib.gdn_forward(*_fwd_args(gdn, s, ws_bytes=ws - 1)) == -6
    assert lib.gdn_forward(*_fwd_args(gdn, s, ws=(1 << 20) + 16, ws_bytes=ws)) == -6
    # unsupported head size, inconsistent chunk count, Hv not a multiple of Hk
    s2 = gdn.make_shape(2, 6, 48, 64, 1, 2, 100, "f32")
    assert lib.gdn_forward(*_fwd_args(gdn, s2, ws_bytes=ws)) == -2
    s3 = gdn.make_shape(2, 6, 64, 64, 1, 1, 100, "f32")
    assert lib.gdn_forward(*_fwd_args(gdn, s3, ws_bytes=ws)) == -1
    s4 = gdn.make_shape(4, 6, 64, 64, 1, 2, 100, "f32")
    assert lib.gdn_forward(*_fwd_args(gdn, s4, ws_bytes=ws)) == -1
    assert lib.gdn_forward(None, *_fwd_args(gdn, s, ws_bytes=ws)[1:]) == -1
    # unknown flags, a backward-only flag, and a keeping forward whose workspace has
    # only the forward's size
    assert lib.gdn_forward(*_fwd_args(gdn, s, ws_bytes=ws, flags=8)) == -1
    # bf16 saved states with fp32 inputs
    assert lib.gdn_forward(*_fwd_args(gdn, s, ws_bytes=ws,
                                      flags=gdn.GDN_FLAG_BF16_SAVED_STATES)) == -2
    assert lib.gdn_forward(*_fwd_args(gdn, s, ws_bytes=ws, flags=gdn.GDN_FLAG_REUSE_FORWARD)) == -1
    assert lib.gdn_forward(*_fwd_args(gdn, s, ws_bytes=ws,
                                      flags=gdn.GDN_FLAG_KEEP_FOR_BACKWARD)) == -6


def test_status_strings(gdn):
    for code, name in [(0, "GDN_OK"), (-1, "GDN_ERR_INVALID_ARG"), (-5, "GDN_ERR_TIMEOUT"),
                       (-7, "GDN_ERR_DEVICE_BOUNDS"), (-8, "GDN_ERR_NOT_KEPT"),
                       (99, "GDN_UNKNOWN_STATUS")]:
        assert gdn.gdn_status_string(code) == name


def test_python_layer_holds_no_cpu_path():
    """The binding only marshals arguments: it must not import the oracle or do math."""
    src = open(os.path.join(ROOT, "gated_deltanet_backward_gb300", "__init__.py")).read()
    assert "oracle" not in src.replace("no fallback", "")
    assert "torch.matmul" not in src and "einsum" not in src


def test_header_is_plain_c(tmp_path):
    """include/gdn.h is a C header: a C99 translation unit that includes it and calls every
    declared entry point through a function pointer compiles cleanly, pedantic."""
    names = sorted(_declared())
    src = tmp_path / "use_gdn.c"
    body = "\n".join("  (void)&%s;" % n for n in names)
    src.write_text('#include "gdn.h"\nint main(void) {\n%s\n  return 0;\n}\n' % body)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-fsyntax-only", "-I", os.path.join(ROOT, "include"), str(src)], check=True)


def test_a_c_program_plans_sizes_and_gets_refusals(gdn, tmp_path):
    """A plain C99 program links libgdn.so and uses its host-only entry points: the chunk
    plan of a varlen batch, the buffer sizes of the 27B-shaped layer, and a forward that
    is refused before any launch (null q), with its status string."""
    src = tmp_path / "plan.c"
    src.write_text(r'''
#include <stdio.h>
#include "gdn.h"
int main(void) {
  const int32_t cu[5] = {0, 64, 64, 200, 201};
  int32_t off[5], nc = -1;
  if (gdn_plan(cu, 4, off, &nc) != GDN_OK) return 1;
  printf("plan %d %d %d %d %d total %d\n", off[0], off[1], off[2], off[3], off[4], nc);
  gdn_shape s = {16, 48, 128, 128, 1, 64, 4096, GDN_DTYPE_BF16, 0.0f,
                 GDN_HEAD_MAP_CONSECUTIVE};
  printf("saved %zu\n", gdn_saved_state_bytes(&s));
  printf("ws %d\n", gdn_workspace_bytes(&s, 1) > gdn_workspace_bytes(&s, 0));
  int rc = gdn_forward(&s, NULL, 10240, NULL, 10240, NULL, 10240, NULL, 48, NULL, 48, NULL,
                       NULL, NULL, NULL, NULL, NULL, 6144, NULL, NULL, NULL, 0, 0u, NULL);
  printf("forward %d %s\n", rc, gdn_status_string(rc));
  return 0;
}
''')
    exe = tmp_path / "plan"
    libdir = os.path.dirname(gdn.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lgdn",
                    "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    assert out[0] == "plan 0 1 1 4 5 total 5"
    assert out[1] == "saved %d" % (64 * 48 * 128 * 128 * 4)
    assert out[2] == "ws 1"
    assert out[3] == "forward -1 GDN_ERR_INVALID_ARG"
