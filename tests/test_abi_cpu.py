"""CPU checks of the C-ABI library: it builds, loads, exports every declared
symbol, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bd_attn.h")


@pytest.fixture(scope="module")
def lib_():
    from packed_sequence_block_gb300 import build, _native
    build.build()
    return _native.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bd_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("bd_doc_ids_from_cu_seqlens", "bd_segment_cu_seqlens", "bd_attn_plan",
              "bd_attn_fwd", "bd_attn_bwd", "bd_get_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib_):
    from packed_sequence_block_gb300 import _native
    for n in declared_symbols():
        assert hasattr(lib_, n), f"{n} missing from libbd_attn.so"
        assert n in _native.SIGNATURES, f"{n} has no Python binding"


def test_status_strings(lib_):
    assert lib_.bd_status_string(0) == b"ok"
    assert b"invalid" in lib_.bd_status_string(1)
    assert lib_.bd_status_string(99) == b"unknown status"
    assert lib_.bd_version() >= 100


def test_sizes_are_host_computed(lib_):
    # plan: 256-aligned sections, grows with the rows
    a = lib_.bd_attn_plan_size(1, 32, 8, 8192, 8192)
    b = lib_.bd_attn_plan_size(2, 32, 8, 8192, 8192)
    assert a > 0 and b > a and a % 256 == 0
    assert lib_.bd_attn_plan_size(0, 1, 1, 1, 1) == 0
    w = lib_.bd_attn_bwd_planned_workspace_size(1, 32, 8, 8192, 8192, 128)
    assert w >= 32 * 8192 * 128 * 4 + 32 * 8192 * 8
    # the single-call workspace holds the plan, the fp16 v, the fp16 copy of O
    # and the backward's accumulator and row terms
    one = lib_.bd_attn_workspace_size(1, 32, 8, 8192, 8192, 128)
    assert one % 256 == 0
    assert one >= (a + lib_.bd_attn_fwd_planned_workspace_size(1, 8, 8192, 128) + w
                   + 2 * 32 * 8192 * 128)
    assert lib_.bd_attn_workspace_size(1, 32, 8, 8192, 8192, 0) == 0


FAKE = 1 << 20  # a non-null, 256-aligned dummy address: never dereferenced on these paths


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, B=1, Hq=4, Hkv=2, L=256, S=256, D=64, seq_start=0,
             scale=0.0, gqa=1, plan=FAKE, plan_bytes=1 << 30, out=FAKE, lse=FAKE, lo=None,
             ws=FAKE, ws_bytes=1 << 30, st=None, stream=None)
    a.update(kw)
    return lib.bd_attn_fwd_planned(a["q"], a["k"], a["v"], a["B"], a["Hq"], a["Hkv"], a["L"], a["S"],
                         a["D"], a["seq_start"], a["scale"], a["gqa"], a["plan"], a["plan_bytes"],
                         a["out"], a["lse"], a["lo"], a["ws"], a["ws_bytes"], a["st"],
                         a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1),
    (dict(D=96), 2),
    (dict(D=0), 1),
    (dict(Hq=3, Hkv=2), 1),
    (dict(gqa=0), 1),
    (dict(seq_start=1), 1),
    (dict(seq_start=-1), 1),
    (dict(L=300), 1),
    (dict(q=FAKE + 8), 1),
    (dict(plan=FAKE + 16), 1),
    (dict(plan_bytes=16), 5),
    (dict(lo=FAKE + 2), 1),
    (dict(ws=None), 1),
    (dict(ws=FAKE + 16), 1),
    (dict(ws_bytes=16), 5),
])
def test_fwd_rejects_bad_arguments(lib_, kw, code):
    assert _fwd(lib_, **kw) == code


def test_bwd_and_plan_reject_bad_arguments(lib_):
    f = lib_.bd_attn_bwd_planned
    args = [FAKE] * 7 + [1, 4, 2, 256, 256, 64, 0, 0.0, 1, FAKE, 1 << 30, FAKE, FAKE, FAKE,
                         FAKE, 1 << 30, None, None]
    bad = list(args)
    bad[12] = 100  # D
    assert f(*bad) == 2
    bad = list(args)
    bad[22] = 8  # workspace too small
    assert f(*bad) == 5
    bad = list(args)
    bad[20] = FAKE + 4  # misaligned dv
    assert f(*bad) == 1
    bad = list(args)
    bad[4] = FAKE + 2  # misaligned out16
    assert f(*bad) == 1
    p = lib_.bd_attn_plan
    assert p(FAKE, FAKE, FAKE, 1, 4, 2, 256, 256, 0, FAKE, 8, None) == 5
    assert p(FAKE, FAKE, FAKE, 1, 4, 2, 256, 200, 0, FAKE, 1 << 30, None) == 1
    assert p(FAKE, FAKE, FAKE, 1, 4, 2, 1 << 22, 1 << 22, 0, FAKE, 1 << 40, None) == 2
    assert lib_.bd_doc_ids_from_cu_seqlens(None, FAKE, 1, 8, FAKE, None, None) == 1
    assert lib_.bd_segment_cu_seqlens(FAKE, 0, 8, FAKE, FAKE, FAKE, None) == 1
    host = ctypes.c_int32(0)
    assert lib_.bd_get_device_status(None, ctypes.addressof(host), None) == 1


def test_layout_entry_points_reject_bad_arguments_on_the_host(lib_):
    f = lib_.bd_doc_ids_from_seq_lens
    assert f(FAKE, 1, 8193, 8, -1000, FAKE, None, None) == 2   # too many documents
    assert f(FAKE, 0, 4, 8, -1000, FAKE, None, None) == 1      # no rows
    assert f(None, 1, 4, 8, -1000, FAKE, None, None) == 1      # lengths missing
    g = lib_.bd_position_ids_from_doc_ids
    assert g(FAKE, 1, 0, FAKE, FAKE, None) == 1
    assert g(FAKE, 1, 8, None, FAKE, None) == 1
    h = lib_.bd_validate_document_positions
    assert h(FAKE, FAKE, 1, 8, None, None, None) == 1
    k = lib_.bd_kv_needed_range
    assert k(FAKE, FAKE, FAKE, 1, 8, 4, 5, FAKE, None, None) == 1  # seq_start + L > S
    assert k(FAKE, FAKE, FAKE, 1, 8, 0, 0, FAKE, None, None) == 1  # L < 1


@pytest.mark.parametrize("p", [1.0, 1.5, -0.1, float("nan")])
def test_dropout_entry_points_reject_bad_p_on_the_host(lib_, p):
    """dropout_p outside [0, 1) is refused before any shape check or launch."""
    f = lib_.bd_attn_fwd_dropout_planned
    assert f(FAKE, FAKE, FAKE, 1, 4, 2, 256, 256, 64, 0, 0.0, 1, FAKE, 1 << 30, FAKE, FAKE, None,
             FAKE, 1 << 30, p, 7, 0, None, None) == 1
    g = lib_.bd_attn_bwd_dropout_planned
    assert g(*([FAKE] * 7), 1, 4, 2, 256, 256, 64, 0, 0.0, 1, FAKE, 1 << 30, FAKE, FAKE, FAKE,
             FAKE, 1 << 30, p, 7, 0, None, None) == 1
    f = lib_.bd_attn_fwd_dropout
    assert f(*([FAKE] * 3), 1, 4, 2, 256, 256, 64, FAKE, FAKE, 0, 0.0, 1, FAKE, FAKE, FAKE,
             1 << 30, p, 7, 0, None, None) == 1
    g = lib_.bd_attn_bwd_dropout
    assert g(*([FAKE] * 6), 1, 4, 2, 256, 256, 64, FAKE, FAKE, 0, 0.0, 1, FAKE, FAKE, FAKE, FAKE,
             1 << 30, p, 7, 0, None, None) == 1


def test_dropout_entry_points_check_shapes_like_the_plain_ones(lib_):
    f = lib_.bd_attn_fwd_dropout_planned
    assert f(FAKE, FAKE, FAKE, 1, 4, 2, 256, 256, 96, 0, 0.0, 1, FAKE, 1 << 30, FAKE, FAKE, None,
             FAKE, 1 << 30, 0.1, 7, 0, None, None) == 2   # D = 96 unsupported
    assert f(FAKE, FAKE, FAKE, 1, 4, 2, 256, 256, 64, 0, 0.0, 1, FAKE, 1 << 30, FAKE, FAKE, None,
             FAKE, 16, 0.1, 7, 0, None, None) == 5        # workspace too small
    g = lib_.bd_attn_bwd_dropout_planned
    assert g(*([FAKE] * 7), 1, 4, 2, 256, 256, 64, 0, 0.0, 1, FAKE, 1 << 30, FAKE, FAKE, FAKE,
             FAKE, 8, 0.1, 7, 0, None, None) == 5         # workspace too small


def _fwd_cu(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, B=1, Hq=4, Hkv=2, L=256, S=256, D=64, cu=FAKE, rp=FAKE,
             seq_start=0, scale=0.0, gqa=1, out=FAKE, lse=FAKE, ws=FAKE, ws_bytes=1 << 30,
             st=None, stream=None)
    a.update(kw)
    return lib.bd_attn_fwd(a["q"], a["k"], a["v"], a["B"], a["Hq"], a["Hkv"], a["L"], a["S"],
                           a["D"], a["cu"], a["rp"], a["seq_start"], a["scale"], a["gqa"],
                           a["out"], a["lse"], a["ws"], a["ws_bytes"], a["st"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(cu=None), 1),
    (dict(rp=None), 1),
    (dict(q=None), 1),
    (dict(D=96), 2),
    (dict(Hq=3, Hkv=2), 1),
    (dict(gqa=0), 1),
    (dict(seq_start=1), 1),
    (dict(L=300), 1),
    (dict(q=FAKE + 8), 1),
    (dict(out=FAKE + 8), 1),
    (dict(ws=None), 1),
    (dict(ws=FAKE + 16), 1),
    (dict(ws_bytes=16), 5),
    (dict(B=1, L=1 << 22, S=1 << 22), 2),
])
def test_single_call_fwd_rejects_bad_arguments(lib_, kw, code):
    assert _fwd_cu(lib_, **kw) == code


def test_single_call_bwd_rejects_bad_arguments(lib_):
    f = lib_.bd_attn_bwd
    args = [FAKE] * 6 + [1, 4, 2, 256, 256, 64, FAKE, FAKE, 0, 0.0, 1, FAKE, FAKE, FAKE, FAKE,
                         1 << 30, None, None]
    bad = list(args)
    bad[11] = 100  # D
    assert f(*bad) == 2
    bad = list(args)
    bad[12] = None  # cu_seqlens
    assert f(*bad) == 1
    bad = list(args)
    bad[21] = 8  # workspace too small
    assert f(*bad) == 5
    bad = list(args)
    bad[19] = FAKE + 4  # misaligned dv
    assert f(*bad) == 1
    st = lib_.bd_attn_bwd_stages
    sargs = args[:-1] + [0, None]
    assert st(*sargs) == 1  # no stage
    sargs = args[:-1] + [8, None]
    assert st(*sargs) == 1  # unknown stage bit


def test_noalloc_limit_matches_the_header():
    from packed_sequence_block_gb300 import _native
    text = open(HEADER).read()
    m = re.search(r"#define\s+BD_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "BD_NOALLOC_SCRATCH_BYTES not found in the header"
    assert _native.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_wait_test_hook_rejects_bad_arguments(lib_):
    f = lib_.bd_test_arm_wait_timeout
    assert f(0, 1000) == 1
    assert f(3, 1000) == 1
    assert f(1, 0) == 1
    assert f(2, 2000001) == 1
