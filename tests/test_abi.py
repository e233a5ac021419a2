"""The C-ABI library builds, loads, exports every symbol include/mx_moe.h
declares, and rejects invalid arguments on the host with the documented status
codes (no GPU needed: validation runs before any CUDA call)."""
from __future__ import annotations

import ctypes as C
import os
import re
import subprocess

import pytest

import expert_ffn_gb300 as mx
from expert_ffn_gb300 import build as mxbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mx_moe.h")

OK, INVALID, ALIGN, UNSUP, WS = 0, -1, -2, -3, -4


@pytest.fixture(scope="module")
def L():
    mxbuild.build()
    return mx.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MX_API\s+[\w\s\*]+?\b(mx_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 10
    assert sorted(mx.EXPORTED) == names
    out = subprocess.run(["nm", "-D", "--defined-only", mxbuild.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, flags=re.M))
    for n in names:
        assert n in exported, n
        assert hasattr(L, n)
    # nothing else leaks out of the library with default visibility
    ours = {s for s in exported if s.startswith("mx_")}
    assert ours == set(names)


def test_strings(L):
    assert L.mx_version().decode().count(".") == 2
    assert L.mx_status_string(-2).decode() == "MX_ERR_ALIGNMENT"


# ------------------------------------------------------------- validation

D, I, E, K, S = 256, 128, 16, 2, 128
FAKE = 0x7F0000000000  # aligned, never dereferenced: validation fails first or T == 0


def layout(**kw):
    import synth
    off, stride = synth.default_layout(D, I)
    lay = mx.make_layout(D, I, E, K, S, stride, off, mx.MX_BF16, 0.5)
    for k, v in kw.items():
        setattr(lay, k, v)
    return lay


def q(rows, cols, bits, base=FAKE):
    return mx.make_qlinear(base, base + 0x100000, base + 0x200000, rows, cols, bits)


def call(L, lay, T=4, x=FAKE + 0x1000000, out=FAKE + 0x2000000, router=None, shared=None, blob=FAKE + 0x3000000,
         idx=FAKE + 0x4000000, w=FAKE + 0x5000000, opt=None, ws=None, ws_bytes=0, ex=True):
    router = router or q(E, D, 8)
    shared = shared or mx.Ffn(q(S, D, 4), q(S, D, 4), q(D, S, 4))
    args = [x, T, C.byref(router), C.byref(shared), blob, C.byref(lay), out, idx, w]
    if ex:
        return L.mx_moe_layer_forward_ex(*args, C.byref(opt) if opt else None, None, ws, ws_bytes)
    return L.mx_moe_layer_forward(*args)


def test_valid_call_with_zero_tokens_is_a_noop(L):
    assert call(L, layout(), T=0) == OK
    assert call(L, layout(), T=0, ex=False) == OK


@pytest.mark.parametrize("field,value,status", [
    ("magic", 0x12345678, INVALID),
    ("version", 4, INVALID),
    ("version", 0, INVALID),
    ("group", 32, UNSUP),
    ("bits", 8, UNSUP),
    ("d_model", 250, UNSUP),
    ("d_expert", 100, UNSUP),
    ("d_shared", 96, UNSUP),
    ("n_experts", 0, UNSUP),
    ("n_experts", 1000, UNSUP),
    ("top_k", 0, INVALID),
    ("top_k", 17, INVALID),
    ("act_dtype", 7, INVALID),
    ("record_stride", 4096 * 14 + 256, ALIGN),
    ("record_stride", 4096, INVALID),
])
def test_layout_rejections(L, field, value, status):
    assert call(L, layout(**{field: value})) == status
    assert call(L, layout(**{field: value}), ex=False) == status
    assert len(L.mx_last_error_string()) > 0


@pytest.mark.parametrize("name", ["gate", "up", "down"])
@pytest.mark.parametrize("which", ["w", "s", "b"])
def test_misaligned_or_outside_sub_offsets(L, name, which):
    lay = layout()
    sub = getattr(lay, name)
    setattr(sub, which, getattr(sub, which) + 8)
    setattr(lay, name, sub)
    assert call(L, lay) == ALIGN
    lay = layout()
    sub = getattr(lay, name)
    setattr(sub, which, lay.record_stride - 16)
    setattr(lay, name, sub)
    assert call(L, lay) == INVALID


def test_pointer_rejections(L):
    lay = layout()
    assert call(L, lay, x=0) == INVALID
    assert call(L, lay, out=0) == INVALID
    assert call(L, lay, idx=0) == INVALID
    assert call(L, lay, blob=0) == INVALID
    assert call(L, lay, x=FAKE + 0x1000008) == ALIGN
    assert call(L, lay, blob=FAKE + 0x3000080) == ALIGN
    assert call(L, lay, w=FAKE + 0x5000002) == ALIGN
    assert call(L, lay, T=-1) == INVALID
    # out overlapping x
    assert call(L, lay, x=FAKE, out=FAKE + 512) == INVALID


def test_matrix_rejections(L):
    lay = layout()
    assert call(L, lay, router=q(E, D, 4)) == UNSUP          # router must be 8-bit
    assert call(L, lay, router=q(E + 1, D, 8)) == INVALID     # wrong expert count
    assert call(L, lay, router=q(E, D, 8, base=FAKE + 4)) == ALIGN
    bad = mx.Ffn(q(S, D, 4), q(S, D, 4), q(S, D, 4))           # transposed down
    assert call(L, lay, shared=bad) == INVALID
    nul = mx.Ffn(q(S, D, 4), mx.make_qlinear(FAKE, 0, FAKE, S, D, 4), q(D, S, 4))
    assert call(L, lay, shared=nul) == INVALID


def test_workspace_rules(L):
    lay = layout()
    need = L.mx_moe_workspace_bytes(C.byref(lay), 4)
    assert need > 0
    assert L.mx_moe_workspace_bytes(C.byref(layout(group=32)), 4) == 0
    assert call(L, lay, ws=FAKE, ws_bytes=need - 1) == WS
    assert call(L, lay, ws=None, ws_bytes=need) == WS
    assert call(L, lay, ws=FAKE + 128, ws_bytes=need) == ALIGN
    # sizes grow with T up to the decode chunk and with the route arrays beyond it
    sizes = [L.mx_moe_workspace_bytes(C.byref(lay), t) for t in (1, 8, 64, 65, 4096)]
    assert sizes == sorted(sizes)


def test_route_rejections(L):
    lay = layout()
    r = q(E, D, 8)
    args = lambda T=4, x=FAKE, ws=FAKE, nb=1 << 30, perm=FAKE: L.mx_moe_route(
        x, T, C.byref(r), C.byref(lay), FAKE, FAKE, FAKE, FAKE, perm, None, None, None, ws, nb)
    assert args(T=0) == OK
    assert args(x=0) == INVALID
    assert args(perm=0) == INVALID
    assert args(nb=16) == WS
    assert args(x=FAKE + 2) == ALIGN


def test_stack_rejections(L):
    lay = layout()
    n = 2
    routers = (mx.QLinear * n)(q(E, D, 8), q(E, D, 8))
    shareds = (mx.Ffn * n)(*[mx.Ffn(q(S, D, 4), q(S, D, 4), q(D, S, 4)) for _ in range(n)])
    blobs = (C.c_void_p * n)(FAKE + 0x3000000, FAKE + 0x3000000)
    lay2 = layout()
    lay2.d_expert = 192
    layouts = (mx.Layout * n)(lay, lay2)
    need = L.mx_moe_stack_workspace_bytes(C.byref(lay), 1)
    rc = L.mx_moe_stack_forward(FAKE, 1, n, routers, shareds, blobs, layouts, FAKE, FAKE, 1e-6, None, FAKE, need)
    assert rc == INVALID and b"layer 1" in L.mx_last_error_string()
    layouts = (mx.Layout * n)(lay, lay)
    rc = L.mx_moe_stack_forward(FAKE, 1, n, routers, shareds, blobs, layouts, FAKE, FAKE, -1.0, None, FAKE, need)
    assert rc == INVALID
    rc = L.mx_moe_stack_forward(FAKE, 1, n, routers, shareds, blobs, layouts, FAKE, FAKE, 1e-6, None, FAKE, need - 1)
    assert rc == WS
    rc = L.mx_moe_stack_forward(FAKE, 0, n, routers, shareds, blobs, layouts, FAKE, FAKE, 1e-6, None, FAKE, need)
    assert rc == OK


# ------------------------------------------------ layout version 2 (optional parts)

LAYOUT_FIELDS = ("magic", "version", "d_model", "d_expert", "n_experts", "top_k", "d_shared", "group", "bits",
                 "record_stride", "gate", "up", "down", "act_dtype", "layer_scalar", "per_expert_scale",
                 "expert_slot", "n_slots", "router_scale", "post_norm", "post_eps", "shared_expert_gate",
                 "down_sb")


def test_layout_struct_matches_the_header(tmp_path):
    """The binding's Layout has the C struct's field offsets and size (a C
    program built against include/mx_moe.h prints them)."""
    src = tmp_path / "off.c"
    body = "".join(f'    printf("%s %zu\\n", "{f}", offsetof(mx_moe_layout, {f}));\n' for f in LAYOUT_FIELDS)
    src.write_text("#include <stddef.h>\n#include <stdio.h>\n#include \"mx_moe.h\"\n"
                   "int main(void) {\n" + body + '    printf("size %zu\\n", sizeof(mx_moe_layout));\n'
                   "    return 0;\n}\n")
    exe = tmp_path / "off"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    for f in LAYOUT_FIELDS:
        assert int(got[f]) == getattr(mx.Layout, f).offset, f
    assert int(got["size"]) == C.sizeof(mx.Layout)


def test_version_one_layout_is_accepted(L):
    lay = layout(version=1)
    assert call(L, lay, T=0) == OK
    # a version-1 caller's struct ends at per_expert_scale: the fields after it are not read
    lay.expert_slot, lay.n_slots = FAKE + 1, -5
    assert call(L, lay, T=0) == OK


@pytest.mark.parametrize("field,value,status", [
    ("expert_slot", FAKE + 1, ALIGN),
    ("router_scale", FAKE + 8, ALIGN),
    ("post_norm", FAKE + 2, ALIGN),
    ("shared_expert_gate", FAKE + 4, ALIGN),
    ("down_sb", FAKE + 8, ALIGN),
])
def test_optional_part_alignment(L, field, value, status):
    lay = layout(**{field: value})
    if field == "expert_slot":
        lay.n_slots = E
    assert call(L, lay) == status


@pytest.mark.parametrize("n_slots", [0, -1, 32768])
def test_slot_table_needs_a_record_count(L, n_slots):
    assert call(L, layout(expert_slot=FAKE, n_slots=n_slots)) == INVALID


def test_post_norm_eps_must_be_nonnegative(L):
    assert call(L, layout(post_norm=FAKE, post_eps=-1e-6)) == INVALID
    assert call(L, layout(post_norm=FAKE, post_eps=float("nan"))) == INVALID


@pytest.mark.parametrize("field", ["router_scale", "post_norm", "shared_expert_gate"])
def test_multi_launch_path_rejects_the_new_parts(L, field):
    """FP32 activations with more than four tokens run the multi-launch decode
    kernels, which do not implement these parts: the call says so before any
    launch."""
    lay = layout(**{field: FAKE}, act_dtype=mx.MX_F32)
    need = L.mx_moe_workspace_bytes(C.byref(lay), 8)
    assert call(L, lay, T=8, ws=FAKE, ws_bytes=need) == UNSUP
    assert b"multi-launch" in L.mx_last_error_string()


def test_route_entry_rejects_router_scale(L):
    lay = layout(router_scale=FAKE)
    r = q(E, D, 8)
    rc = L.mx_moe_route(FAKE, 4, C.byref(r), C.byref(lay), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE,
                        1 << 30)
    assert rc == UNSUP


# ------------------------------------------------ layout version 3 (packed down words)

def test_version_two_layout_is_accepted(L):
    """A version-2 caller's struct ends at shared_expert_gate: down_sb is not read."""
    lay = layout(version=2)
    lay.down_sb = FAKE + 8
    assert call(L, lay, T=0) == OK


def test_down_sb_bytes(L):
    """Column-major (scale | bias << 16) words: every record's I/64 groups of D
    rows, then the shared expert's S/64 groups."""
    lay = layout()
    assert L.mx_moe_down_sb_bytes(C.byref(lay)) == (E * (I // 64) + S // 64) * D * 4
    lay = layout(expert_slot=FAKE, n_slots=5)
    assert L.mx_moe_down_sb_bytes(C.byref(lay)) == (5 * (I // 64) + S // 64) * D * 4
    assert L.mx_moe_down_sb_bytes(C.byref(layout(magic=1))) == 0


def test_pack_down_sb_host_checks(L):
    """Rejections that come before any launch."""
    lay = layout()
    sd = q(D, S, 4)
    out = FAKE + 0x8000000
    assert L.mx_moe_pack_down_sb(C.byref(layout(magic=1)), FAKE, C.byref(sd), out, None) == INVALID
    assert L.mx_moe_pack_down_sb(C.byref(lay), None, C.byref(sd), out, None) == INVALID
    assert L.mx_moe_pack_down_sb(C.byref(lay), FAKE, None, out, None) == INVALID
    assert L.mx_moe_pack_down_sb(C.byref(lay), FAKE, C.byref(sd), None, None) == INVALID
    assert L.mx_moe_pack_down_sb(C.byref(lay), FAKE, C.byref(q(S, D, 4)), out, None) != OK  # transposed shape
    assert L.mx_moe_pack_down_sb(C.byref(lay), FAKE, C.byref(sd), out + 4, None) == ALIGN
    assert L.mx_moe_pack_down_sb(C.byref(lay), FAKE, C.byref(sd), FAKE + 0x1000, None) == INVALID  # inside the blob
    assert len(L.mx_last_error_string()) > 0
