"""The C-ABI library without a GPU: it loads, exports every declared symbol, and rejects bad
arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "strata.h")


@pytest.fixture(scope="module")
def st():
    from int4_grouped_expert_gb300 import build
    build.build()
    import int4_grouped_expert_gb300 as mod
    mod.lib()
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(strata_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("strata_quantize_groups", "strata_route_topk", "strata_moe_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(st):
    lib = ctypes.CDLL(st.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) <= set(st._SIGNATURES)


def test_status_strings(st):
    for i, name in enumerate(st.STATUS_NAMES):
        assert st.strata_status_string(i) == name
    assert st.strata_status_string(99) == "STRATA_ERR_UNKNOWN"
    assert st.strata_version() >= 100


def test_quantize_host_checks(st):
    A = 1 << 12  # a 16-byte aligned fake address: never dereferenced, checks fail first
    assert st.strata_quantize_groups(A, 4, 100, A, A) == 2
    assert st.strata_quantize_groups(A, 4, 256, A, A, group_size=32) == 3
    assert st.strata_quantize_groups(A, 4, 256, A, A, group_size=512) == 3
    assert st.strata_quantize_groups(A, 4, 320, A, A, group_size=256) == 2   # 320 % 256
    assert st.strata_quantize_groups(None, 4, 256, A, A) == 1
    assert st.strata_quantize_groups(A + 2, 4, 256, A, A) == 1
    assert st.strata_quantize_groups(A, -1, 256, A, A) == 2
    assert st.strata_quantize_groups(A, 0, 256, A, A) == 0
    assert st.strata_quantize_groups_bits(A, 4, 256, A, A, bits=2) == 3
    assert st.strata_quantize_groups_bits(A, 4, 256, A, A, bits=16) == 3
    assert st.strata_quantize_groups_bits(A, 4, 256, A, A, group_size=512, bits=8) == 3
    assert st.strata_quantize_groups_bits(A, 4, 100, A, A, bits=8) == 2
    assert st.strata_quantize_groups_bits(A + 2, 4, 256, A, A, bits=8) == 1
    assert st.strata_quantize_groups_bits(A, 0, 256, A, A, bits=8) == 0


def layer(st, **kw):
    A = 1 << 12
    d = dict(H=4096, I=1536, E=288, k=8, has_shared=1, flags=0, w_router=A, bias=None,
             gate_codes=A, gate_scales=A, up_codes=A, up_scales=A, down_codes=A, down_scales=A)
    d.update(kw)
    return st.strata_moe_layer(**d)


def test_workspace_sizes(st):
    s1 = st.strata_moe_workspace_size(layer(st), 1)
    s16 = st.strata_moe_workspace_size(layer(st), 16)
    assert s1 > 0 and s16 > 0          # (tiny batches add partial-sum scratch: no monotonicity)
    assert s16 % 256 == 0 and s1 % 256 == 0
    # h (bf16 [T*k+T, I]) and y (fp32 [T*k+T, H]) dominate
    assert s16 >= 2 * 144 * 1536 + 4 * 144 * 4096
    assert st.strata_moe_workspace_size(layer(st, H=4000), 4) == 0
    assert st.strata_moe_workspace_size(layer(st, k=0), 4) == 0
    assert st.strata_moe_workspace_size(layer(st, E=1024, has_shared=1), 4) == 0
    assert st.strata_route_workspace_size(16, 288, 8) > 0


def test_workspace_follows_the_decode_schedule(st):
    """The decode GEMMs cut their stages into equal ranges per CTA when a batch leaves at most two
    tiles per CTA, and those ranges need two 8 KB partial-sum slots per CTA (2 x 152 SMs). At most
    ((T*k + T)/8 + segments) chunks x 12 (gate/up) or 16 (down) row blocks: on the 288-expert
    layer T <= 4 stays within 2 x 304 tiles, and T = 8 (up to 74 x 16) claims whole tiles with no
    contraction split and needs no slots. On the 128-expert top-4 layer (I = 2048) T = 8 reaches
    exactly 38 x 16 = 608 tiles and takes equal ranges."""
    slots = 2 * 152 * 2 * 8 * 256 * 4
    for T in (1, 2, 4):
        assert st.strata_moe_workspace_size(layer(st), T) >= slots
    assert st.strata_moe_workspace_size(layer(st), 8) < slots
    assert st.strata_moe_workspace_size(layer(st, I=2048, E=128, k=4), 8) >= slots
    assert st.strata_moe_workspace_size(layer(st, I=2048, E=128, k=4), 16) < slots


@pytest.mark.parametrize("kw,expect", [(dict(H=1000), 2), (dict(I=100), 2), (dict(k=9, E=8), 1),
                                       (dict(k=33, E=64), 1), (dict(E=0), 3), (dict(flags=0x10), 1),
                                       (dict(has_shared=2), 1), (dict(gate_codes=None), 1),
                                       (dict(up_codes=(1 << 12) + 8), 1), (dict(bits=3), 3),
                                       (dict(bits=8, flags=0x100), 3)])
def test_forward_host_checks(st, kw, expect):
    A = 1 << 12
    assert st.strata_moe_forward(layer(st, **kw), A, 4, 2 * A, A, 1 << 30) == expect


def test_forward_workspace_and_buffer_checks(st):
    A = 1 << 12
    L = layer(st)
    need = st.strata_moe_workspace_size(L, 4)
    assert st.strata_moe_forward(L, A, 4, 2 * A, A, need - 1) == 4
    assert st.strata_moe_forward(L, A, 4, 2 * A, A + 16, need) == 4      # workspace misaligned
    assert st.strata_moe_forward(L, A, 4, 2 * A, None, need) == 4
    assert st.strata_moe_forward(L, A, 4, A, A, need) == 1               # out aliases x
    assert st.strata_moe_forward(L, A + 8, 4, 2 * A, A, need) == 1       # x misaligned
    assert st.strata_moe_forward(L, A, 0, 2 * A, None, 0) == 0           # empty batch: no-op
    assert st.strata_moe_forward(L, A, -3, 2 * A, A, need) == 2


def test_route_host_checks(st):
    A = 1 << 12
    ws = st.strata_route_workspace_size(8, 16, 2)
    assert st.strata_route_topk(A, A, None, 8, 1000, 16, 2, 0, A, A, workspace=A, ws_bytes=ws) == 2
    assert st.strata_route_topk(A, A, None, 8, 1024, 16, 17, 0, A, A, workspace=A, ws_bytes=ws) == 1
    assert st.strata_route_topk(A, A, None, 8, 1024, 2000, 2, 0, A, A, workspace=A, ws_bytes=ws) == 3
    assert st.strata_route_topk(A, A, None, 8, 1024, 16, 2, 8, A, A, workspace=A, ws_bytes=ws) == 1
    assert st.strata_route_topk(A, A, None, 8, 1024, 16, 2, 0, A, A, counts=A, workspace=A,
                                ws_bytes=ws) == 1                          # partial grouping set
    assert st.strata_route_topk(A, A, None, 8, 1024, 16, 2, 0, A, A, workspace=A, ws_bytes=ws - 1) == 4


def test_status_reads_reject_null(st):
    assert st.strata_read_status(None)[0] == 1
    assert st.strata_workspace_status(None)[0] == 4


def test_stack_host_checks(st):
    A = 1 << 12
    Ls = [layer(st), layer(st)]
    need = st.strata_moe_stack_workspace_size(Ls, 4)
    one = st.strata_moe_workspace_size(layer(st, flags=2), 4)
    assert need >= one + 2 * 4 * 4096 * 2
    assert st.strata_moe_stack_workspace_size([layer(st), layer(st, H=2048)], 4) == 0
    assert st.strata_moe_stack_forward([layer(st), layer(st, H=2048)], A, 4, 2 * A, A, need) == 2
    assert st.strata_moe_stack_forward(Ls, A, 4, 2 * A, A, need - 1) == 4
    assert st.strata_moe_stack_forward(Ls, A, 4, A, A, need) == 1
    assert st.strata_moe_stack_forward(Ls, A, 0, 2 * A, A, need) == 0


def test_padded_forward_host_checks(st):
    A = 1 << 12
    L = layer(st)
    need = st.strata_moe_workspace_size(L, 16)
    assert st.strata_moe_forward_padded(L, A, None, 16, 2 * A, A, need) == 1       # no count
    assert st.strata_moe_forward_padded(L, A, A + 2, 16, 2 * A, A, need) == 1      # misaligned
    assert st.strata_moe_forward_padded(L, A, 3 * A, 0, 2 * A, A, need) == 2       # T_max < 1
    big = st.strata_moe_workspace_size(L, 65)
    assert st.strata_moe_forward_padded(L, A, 3 * A, 65, 2 * A, A, big) == 3       # > fused router
    assert st.strata_moe_forward_padded(layer(st, flags=0x200), A, 3 * A, 16, 2 * A, A, need) == 3
    assert st.strata_moe_forward_padded(layer(st, bits=8), A, 3 * A, 16, 2 * A, A, 1 << 30) == 3
    assert st.strata_moe_forward_padded(L, A, 3 * A, 16, 2 * A, A, need - 1) == 4
    assert st.strata_moe_forward_padded(L, A, 3 * A, 16, A, A, need) == 1          # out aliases x


def test_group_rows_host_checks(st):
    A = 1 << 12
    W = st.GROUP_WORKSPACE_BYTES
    assert st.strata_group_rows(A, -1, 8, 288, A, A, A, A, A, W) == 2
    assert st.strata_group_rows(A, 4, 0, 288, A, A, A, A, A, W) == 1
    assert st.strata_group_rows(A, 4, 33, 288, A, A, A, A, A, W) == 1
    assert st.strata_group_rows(A, 4, 8, 1025, A, A, A, A, A, W) == 1
    assert st.strata_group_rows(A, 4, 8, 288, None, A, A, A, A, W) == 1
    assert st.strata_group_rows(A, 4, 8, 288, A, A, None, A, A, W) == 1
    assert st.strata_group_rows(A + 2, 4, 8, 288, A, A, A, A, A, W) == 1
    assert st.strata_group_rows(A, 4, 8, 288, A, A, A, A, A, W - 1) == 4
    assert st.strata_group_rows(A, 4, 8, 288, A, A, A, A, A + 16, W) == 4


def test_wait_selftest_host_checks(st):
    A = 1 << 12
    assert st.strata_selftest_bounded_waits(None, 1000) == 1
    assert st.strata_selftest_bounded_waits(A + 4, 1000) == 1
    assert st.strata_selftest_bounded_waits(A, 0) == 1
    assert st.strata_selftest_bounded_waits(A, 5_000_000_000) == 1
