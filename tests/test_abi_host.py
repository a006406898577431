"""Host-side checks of the C ABI: the library builds and loads, exports every
symbol the header declares, and its host-only entry points (scheduler,
capacity, sizes, argument validation) behave as documented. No GPU needed:
no call here reaches a kernel."""

import ctypes
import os
import re

import pytest

from w4a16_int4_moe_gb300 import ops

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "w4a16moe.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 13
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(ops.EXPORTED)


def test_status_strings(lib):
    for st in range(7):
        assert ops.status_string(st)
    assert ops.status_string(99) == "unknown status"
    assert ops.w4a16_version() == 122


def test_align_capacity_closed_form(lib):
    # roundup(numel + min(E, numel) * (bm - 1), bm)
    assert ops.w4a16_align_capacity(576 * 8, 48, 16) == ((4608 + 48 * 15 + 15) // 16) * 16
    assert ops.w4a16_align_capacity(6, 3, 4) == 16
    assert ops.w4a16_align_capacity(2, 384, 16) == 32      # min(E, numel) = 2
    assert ops.w4a16_align_capacity(0, 8, 16) == 0
    assert ops.w4a16_align_capacity(-1, 8, 16) == 0


def test_plan_follows_tok_e(lib):
    # decode, 9-15 rows/expert: one block per expert with headroom
    p = ops.w4a16_plan(576, 8, 384, 4096, 7168, 12.0)
    assert p.block_m == 32 and p.bn == 128 and p.bk == 64 and p.swap_ab == 1
    # TP8 T=16: a third of a row per expert
    assert ops.w4a16_plan(16, 8, 384, 512, 7168).block_m == 16
    # prefill above the ~80 rows/expert switch
    assert ops.w4a16_plan(8192, 8, 384, 4096, 7168, 81.3).block_m == 64
    # heavy prefill: 128-row blocks for both GEMMs
    assert ops.w4a16_plan(8192, 8, 48, 4096, 7168, 600.0).block_m == 128
    assert ops.w4a16_plan(8192, 8, 48, 7168, 2048, 600.0).block_m == 128
    for tok_e in (0.3, 5, 12, 40, 80, 81, 150, 400):
        p = ops.w4a16_plan(1024, 8, 48, 4096, 7168, float(tok_e))
        assert 16 <= p.block_m <= 256 and p.block_m % 16 == 0
        assert 4 <= p.stages <= 16 and p.stages % 4 == 0 and p.split_k == 1
        assert 4 <= p.b_stages <= 32 and p.b_stages % 4 == 0
        ops.w4a16_plan_info(p, 7168)  # a plan the GEMM accepts


def test_plan_ring_depths():
    # The deepest rings that fit in 227 KB of shared memory, an activation
    # ring of at least six stages first: blocks of up to 32 rows get 8
    # activation stages (16 k steps) and 16 weight stages; 64-row blocks,
    # whose epilogue stages the whole block (32 KB), get 6 and 8.
    decode = ops.w4a16_plan(576, 8, 48, 4096, 7168, 12.0)
    assert (decode.block_m, decode.b_stages, decode.stages) == (32, 16, 16)
    tp8 = ops.w4a16_plan(16, 8, 384, 512, 7168)
    assert (tp8.block_m, tp8.b_stages, tp8.stages) == (16, 16, 16)
    prefill = ops.w4a16_plan(8192, 8, 48, 4096, 7168, 81.3)
    assert (prefill.block_m, prefill.b_stages, prefill.stages) == (64, 12, 8)
    # 128-row blocks: 4 two-step activation slots (32 KB each) and the 32 KB
    # BF16 staging tile of the early epilogue leave room for 4 weight stages;
    # 256-row blocks: 4 single-step slots (32 KB each), 8 weight stages
    heavy_dn = ops.w4a16_plan(8192, 8, 48, 7168, 2048, 300.0)
    assert (heavy_dn.block_m, heavy_dn.b_stages, heavy_dn.stages) == (128, 8, 4)
    heavy_gu = ops.w4a16_plan(8192, 8, 48, 4096, 7168, 300.0)
    assert (heavy_gu.block_m, heavy_gu.b_stages, heavy_gu.stages) == (128, 8, 4)
    # a 256-row plan set by the caller: 4 single-step slots and 8 weight stages
    big = ops.Plan.from_buffer_copy(heavy_gu)
    big.block_m, big.b_stages, big.stages = 256, 4, 8
    assert ops.w4a16_plan_info(big, 7168).smem_bytes <= 227 * 1024


def test_plan_rejects_bad_sizes(lib):
    p = ops.Plan()
    assert lib.w4a16_plan(0, 8, 0, 1, 1, 0.0, ctypes.byref(p)) == ops.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_plan(4, 8, 4, 1, 1, 0.0, None) == ops.W4A16_ERR_INVALID_ARG


def test_prepack_size_and_unsupported_schemes(lib):
    assert ops.w4a16_prepack_size(48, 4096, 7168) == 48 * 32 * 112 * 4608
    # ragged n pads to whole 128-row tiles, k = 32 mod 64 to a whole k step
    assert ops.w4a16_prepack_size(2, 130, 96) == 2 * 2 * 2 * 4608
    out = ctypes.c_size_t(0)
    # group != 32, k not a multiple of 32, unknown layout: refused at load
    assert lib.w4a16_prepack_size(1, 128, 128, 64, 0, ctypes.byref(out)) == ops.W4A16_ERR_UNSUPPORTED
    assert lib.w4a16_prepack_size(1, 128, 100, 32, 0, ctypes.byref(out)) == ops.W4A16_ERR_UNSUPPORTED
    assert lib.w4a16_prepack_size(1, 128, 128, 32, 7, ctypes.byref(out)) == ops.W4A16_ERR_UNSUPPORTED
    assert lib.w4a16_prepack(None, None, 1, 128, 128, 16, 0, None, 0, None) == ops.W4A16_ERR_UNSUPPORTED
    # the interleaved gate/up layout needs whole 128-row tiles (n = 2I, I % 64 == 0)
    glu = ops.W4A16_LAYOUT_KTILE64_GLU16
    assert ops.w4a16_prepack_size(2, 512, 256, layout=glu) == ops.w4a16_prepack_size(2, 512, 256)
    assert lib.w4a16_prepack_size(1, 192, 128, 32, glu, ctypes.byref(out)) == ops.W4A16_ERR_UNSUPPORTED
    assert lib.w4a16_prepack(None, None, 1, 128, 128, 32, 0, None, 0, None) == ops.W4A16_ERR_INVALID_ARG


def test_gemm_argument_checks_before_any_launch(lib):
    plan = ops.w4a16_plan(64, 2, 8, 1024, 512)
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: checks fail first
    args = dict(mode=ops.W4A16_GATE_UP, packed=fake, E=8, n=1024, k=512, a=fake, tokens=64,
                topk=2, sid=fake, eid=fake, ntp=fake, cap=256, w=None, out=fake, flags=0,
                ws=fake, wsb=1 << 30)

    def call(**kw):
        a = dict(args, **kw)
        return lib.w4a16_moe_indexed_gemm(a["mode"], a["packed"], a["E"], a["n"], a["k"], a["a"],
                                          a["tokens"], a["topk"], a["sid"], a["eid"], a["ntp"],
                                          a["cap"], a["w"], a["out"], a["flags"], ctypes.byref(plan),
                                          a["ws"], a["wsb"], None)
    assert call(mode=7) == ops.W4A16_ERR_INVALID_ARG
    assert call(k=500) == ops.W4A16_ERR_UNSUPPORTED           # k % 32 != 0
    assert call(mode=ops.W4A16_DOWN) == ops.W4A16_ERR_INVALID_ARG  # no top-k weights
    assert call(ws=None) == ops.W4A16_ERR_WORKSPACE
    assert call(wsb=16) == ops.W4A16_ERR_WORKSPACE
    # the workspace holds the routed rows: 256 status bytes + cap x roundup(k, 64) BF16
    need = ops.w4a16_workspace_size(plan, 256, 512)
    assert need == 256 + 256 * 512 * 2
    assert ops.w4a16_workspace_size(plan, 256, 480) == 256 + 256 * 512 * 2
    assert ops.w4a16_workspace_size(plan, 0, 512) == 256
    assert call(wsb=need - 1) == ops.W4A16_ERR_WORKSPACE
    assert call(cap=250) == ops.W4A16_ERR_INVALID_ARG          # not a multiple of block_m
    assert call(flags=64) == ops.W4A16_ERR_INVALID_ARG
    # the deterministic sum is a DOWN option, and needs its own workspace part
    assert call(flags=ops.W4A16_FLAG_DETERMINISTIC) == ops.W4A16_ERR_INVALID_ARG
    det_w = ctypes.c_void_p(1 << 20)
    assert call(mode=ops.W4A16_DOWN, w=det_w, flags=ops.W4A16_FLAG_DETERMINISTIC,
                wsb=need) == ops.W4A16_ERR_WORKSPACE
    det = ops.w4a16_deterministic_bytes(256, 1024, 128)
    assert det == 256 * 1024 * 4 + 512   # rows, then 128 int32 positions (256-byte units)
    assert ops.w4a16_deterministic_bytes(-1, 1024, 128) == 0
    assert call(out=ctypes.c_void_p((1 << 20) + 2)) == ops.W4A16_ERR_INVALID_ARG  # misaligned
    bad = ops.Plan.from_buffer_copy(plan)
    bad.block_m = 24
    assert lib.w4a16_moe_indexed_gemm(0, fake, 8, 1024, 512, fake, 64, 2, fake, fake, fake, 240,
                                      None, fake, 0, ctypes.byref(bad), fake, 1 << 30, None) \
        == ops.W4A16_ERR_INVALID_ARG
    bad = ops.Plan.from_buffer_copy(plan)
    bad.block_m = 144   # above the largest block (two partial accumulators must fit in TMEM)
    assert lib.w4a16_moe_indexed_gemm(0, fake, 8, 1024, 512, fake, 64, 2, fake, fake, fake, 288,
                                      None, fake, 0, ctypes.byref(bad), fake, 1 << 30, None) \
        == ops.W4A16_ERR_INVALID_ARG
    for field, value in (("stages", 3), ("stages", 17), ("b_stages", 6), ("b_stages", 10)):
        bad = ops.Plan.from_buffer_copy(plan)
        setattr(bad, field, value)   # weight ring below one stage per warpgroup; odd B stages
        assert lib.w4a16_moe_indexed_gemm(0, fake, 8, 1024, 512, fake, 64, 2, fake, fake, fake,
                                          256, None, fake, 0, ctypes.byref(bad), fake, 1 << 30,
                                          None) == ops.W4A16_ERR_INVALID_ARG, field
    # the fused activation needs the interleaved packing named in the plan, and
    # the other modes the plain one
    glu_plan = ops.Plan.from_buffer_copy(plan)
    glu_plan.layout = ops.W4A16_LAYOUT_KTILE64_GLU16
    assert call(mode=ops.W4A16_GATE_UP_SILU) == ops.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, fake, 8, 1024, 512, fake, 64, 2, fake,
                                      fake, fake, 256, None, fake, 0, ctypes.byref(glu_plan),
                                      fake, 1 << 30, None) == ops.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP_SILU, fake, 8, 1000, 512, fake, 64, 2,
                                      fake, fake, fake, 256, None, fake, 0,
                                      ctypes.byref(glu_plan), fake, 1 << 30, None) \
        == ops.W4A16_ERR_UNSUPPORTED   # n not whole 128-row tiles
    bad = ops.Plan.from_buffer_copy(plan)
    bad.split_k = 2
    assert lib.w4a16_moe_indexed_gemm(0, fake, 8, 1024, 512, fake, 64, 2, fake, fake, fake, 256,
                                      None, fake, 0, ctypes.byref(bad), fake, 1 << 30, None) \
        == ops.W4A16_ERR_INVALID_ARG


def test_empty_calls_accept_null_arrays_and_enqueue_nothing(lib):
    # no tokens, capacity 0: the zero-element arrays may be NULL and the calls
    # return before any CUDA call (so this runs without a GPU); a NULL array
    # that has elements is refused
    fake = ctypes.c_void_p(1 << 20)
    plan = ops.w4a16_plan(64, 2, 8, 1024, 512, 0.0)
    for mode in (ops.W4A16_GATE_UP, ops.W4A16_DOWN):
        assert lib.w4a16_moe_indexed_gemm(mode, fake, 8, 1024, 512, None, 0, 2, None, None, fake,
                                          0, None, None, 0, ctypes.byref(plan), fake, 1 << 20,
                                          None) == ops.W4A16_OK
    assert lib.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, fake, 8, 1024, 512, fake, 64, 2, fake,
                                      fake, fake, 256, None, None, 0, ctypes.byref(plan), fake,
                                      1 << 30, None) == ops.W4A16_ERR_INVALID_ARG   # no output
    assert lib.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, fake, 8, 1024, 512, fake, 64, 2, None,
                                      fake, fake, 256, None, fake, 0, ctypes.byref(plan), fake,
                                      1 << 30, None) == ops.W4A16_ERR_INVALID_ARG   # no sorted_ids
    assert lib.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, fake, 8, 1024, 512, None, 0, 2, None,
                                      None, None, 0, None, None, 0, ctypes.byref(plan), fake,
                                      1 << 20, None) == ops.W4A16_ERR_INVALID_ARG   # ntp NULL
    gplan = ops.w4a16_grouped_plan(ops.W4A16_GROUPED_CONTIGUOUS, 128, 1024, 512)
    assert lib.w4a16_moe_grouped_gemm(ops.W4A16_GROUPED_CONTIGUOUS, fake, 8, 1024, 512, None, 0,
                                      None, 0, None, 0, ctypes.byref(gplan), fake, 256,
                                      None) == ops.W4A16_OK
    assert lib.w4a16_moe_grouped_gemm(ops.W4A16_GROUPED_MASKED, fake, 8, 1024, 512, None, 0,
                                      fake, 0, None, 0, ctypes.byref(gplan), fake, 256,
                                      None) == ops.W4A16_OK
    assert lib.w4a16_moe_grouped_gemm(ops.W4A16_GROUPED_MASKED, fake, 8, 1024, 512, None, 0,
                                      None, 0, None, 0, ctypes.byref(gplan), fake, 256,
                                      None) == ops.W4A16_ERR_INVALID_ARG   # masked_m [E] NULL
    glu = ops.w4a16_plan(64, 2, 8, 1024, 512, 0.0)
    glu.layout = ops.W4A16_LAYOUT_KTILE64_GLU16
    assert lib.w4a16_moe_layer(fake, fake, 8, 512, 512, None, 0, 2, None, None, fake, 0, None,
                               None, 0, ctypes.byref(glu), fake, 256, None) == ops.W4A16_OK
    assert lib.w4a16_moe_layer(fake, fake, 8, 512, 512, fake, 64, 2, fake, fake, fake, 256, fake,
                               None, 0, ctypes.byref(glu), fake, 1 << 30,
                               None) == ops.W4A16_ERR_INVALID_ARG   # no output
    assert lib.w4a16_silu_and_mul(None, 0, 512, None, None) == ops.W4A16_OK


def test_row_counts_of_2_pow_30_are_refused(lib):
    # flattened routed rows (tokens x topk) index the routing as int32 with
    # room for the sentinel: 2^30 rows and above are refused before any
    # CUDA call
    fake = ctypes.c_void_p(1 << 20)
    plan = ops.w4a16_plan(64, 2, 8, 1024, 512, 0.0)
    big = 1 << 27   # x 8 = 2^30
    assert lib.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, fake, 8, 1024, 512, fake, big, 8, fake,
                                      fake, fake, 256, None, fake, 0, ctypes.byref(plan), fake,
                                      1 << 40, None) == ops.W4A16_ERR_UNSUPPORTED
    assert lib.w4a16_moe_align_block_size(fake, big, 8, 8, 16, 1 << 30, fake, fake, fake,
                                          None) == ops.W4A16_ERR_UNSUPPORTED


def test_grouped_and_align_argument_checks(lib):
    fake = ctypes.c_void_p(1 << 20)
    plan = ops.w4a16_plan(32, 1, 1, 256, 256, 32.0)
    assert lib.w4a16_moe_grouped_gemm(5, fake, 4, 256, 256, fake, 128, fake, 16, fake, 0,
                                      ctypes.byref(plan), fake, 256, None) == ops.W4A16_ERR_INVALID_ARG
    bad = ops.Plan.from_buffer_copy(plan)
    bad.block_m = 48   # does not divide the 128-row expert alignment
    assert lib.w4a16_moe_grouped_gemm(0, fake, 4, 256, 256, fake, 144, fake, 16, fake, 0,
                                      ctypes.byref(bad), fake, 256, None) == ops.W4A16_ERR_INVALID_ARG
    # align: capacity too small, not a multiple of block_m, too many experts
    assert lib.w4a16_moe_align_block_size(fake, 64, 2, 8, 16, 64, fake, fake, fake, None) \
        == ops.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_moe_align_block_size(fake, 64, 2, 8, 16, 250, fake, fake, fake, None) \
        == ops.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_moe_align_block_size(fake, 64, 2, 2000, 16, 1 << 16, fake, fake, fake, None) \
        == ops.W4A16_ERR_UNSUPPORTED
    assert lib.w4a16_silu_and_mul(fake, 4, 12, fake, None) == ops.W4A16_ERR_INVALID_ARG


def test_route_align_and_layer_argument_checks(lib):
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: checks fail first

    def route(**kw):
        a = dict(logits=fake, dtype=ops.W4A16_DTYPE_F32, tokens=64, experts=384, topk=8,
                 renorm=1, offset=0, local=48, bm=16, cap=16 * 100, arrivals=fake)
        a.update(kw)
        return lib.w4a16_moe_route_align(a["logits"], a["dtype"], a["tokens"], a["experts"],
                                         a["topk"], a["renorm"], a["offset"], a["local"], a["bm"],
                                         a["cap"], fake, fake, fake, fake, fake, a["arrivals"],
                                         None)
    assert route(dtype=5) == ops.W4A16_ERR_INVALID_ARG
    assert route(arrivals=None) == ops.W4A16_ERR_INVALID_ARG      # the counter is required
    assert route(cap=16 * 100 + 8) == ops.W4A16_ERR_INVALID_ARG   # not whole blocks
    assert route(cap=16) == ops.W4A16_ERR_INVALID_ARG             # below the bound
    assert route(local=0) == ops.W4A16_ERR_INVALID_ARG
    assert route(experts=1025) == ops.W4A16_ERR_UNSUPPORTED
    assert route(topk=33) == ops.W4A16_ERR_UNSUPPORTED
    assert route(local=1025, cap=1 << 20) == ops.W4A16_ERR_UNSUPPORTED
    assert route(tokens=64, logits=None) == ops.W4A16_ERR_INVALID_ARG

    plan = ops.w4a16_plan(576, 8, 48, 4096, 7168, 12.0)
    glu = ops.Plan.from_buffer_copy(plan)
    glu.layout = ops.W4A16_LAYOUT_KTILE64_GLU16
    cap = ops.w4a16_align_capacity(576 * 8, 48, glu.block_m)
    need = ops.w4a16_layer_workspace_size(glu, cap, 7168, 2048)

    def layer(p=glu, **kw):
        a = dict(hidden=7168, inter=2048, x=fake, cap=cap, w=fake, out=fake, flags=0,
                 ws=fake, wsb=need)
        a.update(kw)
        return lib.w4a16_moe_layer(fake, fake, 48, a["hidden"], a["inter"], a["x"], 576, 8,
                                   fake, fake, fake, a["cap"], a["w"], a["out"], a["flags"],
                                   ctypes.byref(p), a["ws"], a["wsb"], None)
    assert layer(p=plan) == ops.W4A16_ERR_INVALID_ARG            # gate_up not GLU16-packed
    pair = ops.Plan.from_buffer_copy(glu)
    pair.cta_pair = 1
    assert layer(p=pair) == ops.W4A16_ERR_INVALID_ARG            # the layer runs unpaired
    assert layer(inter=2000) == ops.W4A16_ERR_UNSUPPORTED        # inter % 64
    assert layer(hidden=7100) == ops.W4A16_ERR_UNSUPPORTED       # hidden % 32
    assert layer(w=None) == ops.W4A16_ERR_INVALID_ARG            # top-k weights required
    assert layer(flags=ops.W4A16_FLAG_DETERMINISTIC) == ops.W4A16_ERR_INVALID_ARG
    assert layer(cap=cap + 8) == ops.W4A16_ERR_INVALID_ARG       # not whole blocks
    assert layer(out=ctypes.c_void_p((1 << 20) + 4)) == ops.W4A16_ERR_INVALID_ARG
    assert layer(wsb=need - 1) == ops.W4A16_ERR_WORKSPACE
    assert layer(ws=None) == ops.W4A16_ERR_WORKSPACE
    # status words, both routed-row buffers, one counter per routing block
    assert need >= 256 + cap * 7168 * 2 + cap * 2048 * 2 + (cap // glu.block_m) * 4


def test_product_path_has_no_cpu_fallback():
    # The package never imports the oracle; a missing library is an error.
    import w4a16_int4_moe_gb300 as pkg
    root = os.path.dirname(pkg.__file__)
    for dirpath, _, files in os.walk(root):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
    saved = ops._lib
    ops._lib = None
    try:
        with pytest.raises(RuntimeError):
            ops.load_library("/nonexistent/libw4a16moe.so")
    finally:
        ops._lib = saved


def test_header_is_plain_c():
    # the boundary header compiles as C (and C++) on its own
    import shutil
    import subprocess
    header = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "include", "w4a16moe.h")
    for cc, lang in (("gcc", "c"), ("g++", "c++")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not installed")
        r = subprocess.run([cc, "-fsyntax-only", "-Wall", "-Werror", "-x", lang, header],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_noalloc_refuses_a_workspace_beyond_its_array(lib):
    # the built-in array holds 32 MiB: at k = 7168 (14336 B per routed row
    # after the 256 status bytes) a routing capacity of 2340 rows fits and
    # 2341 does not. Capacity 2340 is not a multiple of block_m 32, so the
    # call that passes the size check is refused right after it, before any
    # CUDA call; nothing is launched with these fake pointers.
    import ctypes
    plan = ops.w4a16_plan(64, 8, 48, 4096, 7168)
    plan.block_m = 32
    fake = ctypes.c_void_p(1 << 20)

    def call(capacity):
        return lib.w4a16_moe_indexed_gemm_noalloc(0, fake, 48, 4096, 7168, fake, 64, 8, fake,
                                                  fake, fake, capacity, None, fake, 0,
                                                  ctypes.byref(plan), None)
    assert ops.w4a16_workspace_size(plan, 2340, 7168) <= 32 << 20
    assert ops.w4a16_workspace_size(plan, 2341, 7168) > 32 << 20
    assert call(2341) == ops.W4A16_ERR_WORKSPACE
    assert call(2340) == ops.W4A16_ERR_INVALID_ARG
