"""The C-ABI library on the CPU: it builds, loads, exports every entry point
declared in include/moe_abi.h, and validates arguments on the host (no kernel
is launched by these tests)."""
import ctypes
import os
import re

import pytest

import routing_dispatch_expert_router_gb300.binding as B
from routing_dispatch_expert_router_gb300.build import build
from workloads import DSV3, DSV3_FP8, MIXTRAL, QWEN3, TINY, MoEShape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "moe_abi.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 15
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.ENTRY_POINTS) == names


def test_query_sizes_worst_case_rows():
    s = B.moe_query_sizes(MIXTRAL)
    assert s.rows_max == 4096 * 2 + 8 * 127 and s.groups == 8 and s.capacity == 0
    s = B.moe_query_sizes(DSV3)
    assert s.rows_max == 8192 * 8 + 256 * 127 + 8192 and s.groups == 257
    s = B.moe_query_sizes(QWEN3)
    assert s.rows_max == 16384 * 8 + 128 * 127
    s = B.moe_query_sizes(TINY)
    assert s.rows_max == 512 + 8 * 127
    s = B.moe_query_sizes(MoEShape("c", T=16384, H=128, E=256, k=8, F=128, capacity_factor=1.25))
    assert s.capacity == 640 and s.rows_max == 256 * 640
    assert s.scratch_bytes >= 4096 + 64 * 256 * 4


@pytest.mark.parametrize("bad", [
    dict(H=100), dict(F=200), dict(k=0), dict(k=9), dict(E=300), dict(k=5, E=4),
    dict(n_groups=3), dict(n_groups=8, topk_groups=0), dict(n_groups=4, topk_groups=1, k=3, E=8),
    dict(row_align=64), dict(capacity_factor=-1.0), dict(score_fn=7), dict(T=-1),
    dict(n_shared=5),
])
def test_invalid_configs_rejected(bad):
    with pytest.raises(B.MoEError) as e:
        B.moe_query_sizes(TINY.with_(**bad))
    assert e.value.code == 1


def test_fp8_scratch_holds_the_quantised_operands():
    s = B.moe_query_sizes(DSV3_FP8)
    G, R, H, F = 256, 256 * 640, 7168, 2048

    def atoms(rows, K):        # one 512-byte scale atom per 128 rows and 4 K blocks of 128
        return rows // 128 * -(-K // 512) * 512

    # E4M3 weights with their scale atoms for both orientations (forward, data gradient)
    weights = G * 2 * F * H + G * H * F + atoms(G * 2 * F, H) + atoms(G * H, 2 * F) + \
        atoms(G * H, F) + atoms(G * F, H)
    # E4M3 x_perm, h, dO, dGU (1x128 slices) with atoms; the same four in 128x1
    # slices (atoms: the columns as rows, the buffer's row blocks as K)
    acts = R * H + R * F + R * H + R * 2 * F + atoms(R, H) + atoms(R, F) + atoms(R, H) + \
        atoms(R, 2 * F) + R * H + R * F + R * 2 * F + R * H + atoms(H, R) + atoms(F, R) + \
        atoms(2 * F, R) + atoms(H, R)
    quantised = weights + acts
    # the tensor-core router's region (E % 128 == 0): the larger of W_r as three
    # bf16 parts (forward) and dlogits as three bf16 parts plus the chunk sums of
    # dW_r^T over 1024-token chunks (backward)
    T, E = 16384, 256
    router_split = max(E * 3 * H * 2, 3 * T * E * 2 + (T // 1024) * H * E * 4)
    assert s.capacity == 640 and s.rows_max == R
    assert quantised + router_split <= s.scratch_bytes <= quantised + router_split + (1 << 20)
    with pytest.raises(B.MoEError) as e:           # shared experts: not in FP8 mode
        B.moe_query_sizes(DSV3_FP8.with_(n_shared=1))
    assert e.value.code == 2
    with pytest.raises(B.MoEError) as e:           # the FP8 GEMM tiles: H, F multiples of 256
        B.moe_query_sizes(DSV3_FP8.with_(H=7168 + 128))
    assert e.value.code == 2
    with pytest.raises(B.MoEError) as e:
        B.moe_query_sizes(DSV3_FP8.with_(dtype=7))
    assert e.value.code == 1


def test_mxfp8_scratch_holds_both_weight_forms():
    """MXFP8: the weights in two E4M3 forms and one scale byte per 32 elements
    (atoms of 128 rows x one 128-wide K block) for weights and activations."""
    mx = DSV3_FP8.with_(dtype=2)
    s = B.moe_query_sizes(mx)
    G, R, H, F = 256, 256 * 640, 7168, 2048
    sfb = lambda rows, K: rows * K // 32          # noqa: E731
    weights = 2 * (G * 2 * F * H + G * H * F) + sfb(G * 2 * F, H) + sfb(G * H, 2 * F) + \
        sfb(G * H, F) + sfb(G * F, H)
    acts = 2 * (R * H + R * F + R * H + R * 2 * F) + sfb(R, H) + sfb(R, F) + sfb(R, H) + \
        sfb(R, 2 * F) + sfb(H, R) + sfb(F, R) + sfb(2 * F, R) + sfb(H, R)
    T, E = 16384, 256
    router_split = max(E * 3 * H * 2, 3 * T * E * 2 + (T // 1024) * H * E * 4)
    assert s.rows_max == R
    assert weights + acts + router_split <= s.scratch_bytes <= weights + acts + router_split + (1 << 20)
    # same restrictions as the block recipe
    with pytest.raises(B.MoEError) as e:
        B.moe_query_sizes(mx.with_(n_shared=1))
    assert e.value.code == 2
    with pytest.raises(B.MoEError) as e:
        B.moe_query_sizes(mx.with_(weights_in_expert=1))
    assert e.value.code == 2


def test_null_and_misaligned_pointers_rejected_before_launch():
    cfg = B.config(TINY)
    lib = B.lib()
    vp = ctypes.c_void_p
    rc = lib.moe_route(ctypes.byref(cfg), vp(None), vp(4096), vp(None), vp(4096), vp(4096),
                       vp(4096), vp(4096), vp(None))
    assert rc == 1
    rc = lib.moe_unpermute(ctypes.byref(cfg), vp(4096 + 8), vp(4096), vp(4096), vp(4096),
                           vp(4096), vp(None))
    assert rc == 1
    rc = lib.moe_layer_fwd(ctypes.byref(cfg), vp(None), vp(4096), vp(4096), vp(None), vp(4096),
                           vp(None))
    assert rc == 1


def test_aux_loss_entry_points_reject_bad_arguments_before_launch():
    """Host-side checks of the load-balancing loss calls (no device work):
    a NULL counts output, a dlogits buffer off 16 bytes, a non-finite
    coefficient or gradient scale."""
    cfg = B.config(TINY)
    lib = B.lib()
    vp, f = ctypes.c_void_p, ctypes.c_float
    ok = vp(4096)
    rc = lib.moe_route_aux(ctypes.byref(cfg), ok, vp(None), ok, f(0.01), f(1e-3), vp(None), ok,
                           ok, vp(None), ok, vp(None))
    assert rc == 1
    rc = lib.moe_route_aux(ctypes.byref(cfg), ok, vp(None), ok, f(float("nan")), f(1e-3), ok, ok,
                           ok, vp(None), ok, vp(None))
    assert rc == 1
    rc = lib.moe_route_aux_bwd(ctypes.byref(cfg), ok, ok, vp(None), ok, ok, f(0.01), f(1.0),
                               vp(4096 + 4), ok, ok, ok, vp(None))
    assert rc == 1
    rc = lib.moe_route_aux_bwd(ctypes.byref(cfg), ok, ok, vp(None), ok, ok, f(0.01),
                               f(float("inf")), ok, ok, ok, ok, vp(None))
    assert rc == 1


def test_status_strings():
    for code in range(8):
        assert B.status_string(code)
    assert "unknown" in B.status_string(99)


def test_noalloc_dispatch_refuses_the_fp8_configuration_before_launch():
    """In the FP8 configuration the dispatch also writes x_perm's E4M3 form
    into the caller's scratch, which the no-scratch entry point cannot take."""
    cfg = B.config(DSV3_FP8)
    vp = ctypes.c_void_p
    ok = vp(4096)
    rc = B.lib().moe_permute_noalloc(ctypes.byref(cfg), ok, ok, ok, ok, ok, ok, ok, ok, ok,
                                     vp(None))
    assert rc == 2                 # MOE_ERR_UNSUPPORTED


def test_reordered_layer_configuration_checks():
    """weights_in_expert: 0 or 1, bf16 mode only; its region of scratch holds
    one fp32 weight per permuted row and one fp32 partial per row and FC2
    data-gradient tile."""
    base = B.moe_query_sizes(MIXTRAL).scratch_bytes
    s = B.moe_query_sizes(MIXTRAL.with_(weights_in_expert=1))
    R = s.rows_max
    assert s.scratch_bytes - base >= R * 4 + R * (14336 // 256) * 4
    with pytest.raises(B.MoEError) as e:
        B.moe_query_sizes(MIXTRAL.with_(weights_in_expert=2))
    assert e.value.code == 1
    with pytest.raises(B.MoEError) as e:
        B.moe_query_sizes(DSV3_FP8.with_(weights_in_expert=1))
    assert e.value.code == 2


def test_paged_stash_configuration_checks():
    """stash_pool_pages: the table length moe_query_sizes reports, the pool's
    range, the layer calls' pointer checks and the per-stage entry points'
    refusal (their buffers are the layer's own R rows) -- all before any launch."""
    s = B.moe_query_sizes(DSV3_FP8)
    assert s.stash_table_len == s.rows_max // 128 + 2
    cfg = B.config(TINY)
    lib = B.lib()
    vp = ctypes.c_void_p
    ok = vp(4096)
    for bad in (-1, (1 << 24)):
        cfg.stash_pool_pages = bad
        sz = B.MoESizes()
        assert lib.moe_query_sizes(ctypes.byref(cfg), ctypes.byref(sz)) == 1
    cfg.stash_pool_pages = 16
    # per-stage entry points: MOE_ERR_UNSUPPORTED with a pool configuration
    assert lib.moe_permute(ctypes.byref(cfg), ok, ok, ok, ok, ok, ok, ok, ok, ok, ok,
                           vp(None)) == 2
    assert lib.moe_grouped_ffn_fwd(ctypes.byref(cfg), ok, ok, ok, ok, ok, ok, ok, ok, ok,
                                   vp(None)) == 2
    assert lib.moe_unpermute(ctypes.byref(cfg), ok, ok, ok, ok, ok, vp(None)) == 2
    # the layer forward wants the page table and the pool counter
    fs = B.MoEFwdState(**{n: 4096 for n in B.FWD_FIELDS})
    P = B.MoEParams(W_r=4096, bias=None, W13=4096, W2=4096)
    assert lib.moe_layer_fwd(ctypes.byref(cfg), ctypes.byref(P), ok, ok, ctypes.byref(fs), ok,
                             vp(None)) == 1
    # releasing needs a pool
    cfg.stash_pool_pages = 0
    fs.stash_table, fs.stash_top = 4096, 4096
    assert lib.moe_stash_release(ctypes.byref(cfg), ctypes.byref(fs), vp(None)) == 1


def test_stash_pool_binding_guards():
    """A pool has at least one page, and a pool's tensors are only handed to a
    configuration that says it uses that pool (else the library would take
    them for the layer's own R-row buffers)."""
    cfg = B.config(TINY)
    with pytest.raises(ValueError):
        B.alloc_stash_pool(cfg, 0, device="cpu")
    pool = B.alloc_stash_pool(cfg, 3, device="cpu")
    assert pool.tensors["x_perm"].shape == (4 * 128, TINY.H)
    with pytest.raises(ValueError):
        B.alloc_buffers(cfg, "cpu", backward=False, pool=pool)      # cfg has no pool
    cfg.stash_pool_pages = 3
    bufs = B.alloc_buffers(cfg, "cpu", backward=False, pool=pool)
    assert bufs.fwd["x_perm"].data_ptr() == pool.tensors["x_perm"].data_ptr()
    assert bufs.fwd["stash_table"].numel() == bufs.sizes.stash_table_len
