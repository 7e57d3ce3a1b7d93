"""Host-side tests of the C ABI: the library loads, exports every declared symbol, and
returns the documented status code for each descriptor/argument rule without touching
a GPU.  Rules: "2 . Le Tensor Memory Accelerator" 2.3 (16-byte base, 16-byte-multiple
strides, box width limited by the swizzle; violations are silent on the hardware, so
the library must catch them); "H100 . cuTensorMap (TMA descriptor)" 8-9 (rank <= 5,
dims in 1..2^32, boxDim in 1..256)."""
import ctypes

import pytest

from tma_pipelined_tensor_gb300 import build as tgbuild
from tma_pipelined_tensor_gb300 import tg


@pytest.fixture(scope="module", autouse=True)
def _built():
    tgbuild.build()


def test_library_exports_every_declared_function():
    names = tg.declared_functions()
    expected = {"tg_status_string", "tg_status_sync", "tg_status_detail", "gemm_bf16",
                "gemm_bf16_ex", "tg_gemm_config_default", "tg_gemm_plan_for", "tma_validate",
                "tma_tile_copy_image_bytes", "tma_tile_copy", "tma_tile_copy_ex",
                "gemm_bf16_noalloc", "tma_validate_nd", "tma_tile_copy_nd_image_bytes",
                "tma_tile_copy_nd"}
    assert expected <= set(names), names
    L = tg.lib()
    for n in names:
        assert hasattr(L, n), n


def test_status_strings():
    for code, name in [(0, "TG_OK"), (1, "TG_ERR_INVALID_VALUE"), (2, "TG_ERR_MISALIGNED"),
                       (3, "TG_ERR_UNSUPPORTED"), (4, "TG_ERR_BUFFER_TOO_SMALL"),
                       (5, "TG_ERR_CUDA"), (6, "TG_ERR_NO_DRIVER_SYMBOL"),
                       (7, "TG_ERR_DEVICE_TIMEOUT"), (99, "TG_ERR_UNKNOWN")]:
        assert tg.tg_status_string(code) == name


def test_config_defaults():
    c = tg.tg_gemm_config_default()
    assert (c.stages, c.cluster, c.tile_n, c.mma) == (0, 0, 0, 0)   # chosen per problem
    assert c.group_m == 16
    # the default struct and a NULL config plan the same launch
    for shape in ((8192, 8192, 8192), (1024, 4096, 16384), (16384, 4096, 1024), (3000, 5000, 2056)):
        st1, p1 = tg.tg_gemm_plan_for(*shape, tg.TG_C_BF16, c, 152)
        st2, p2 = tg.tg_gemm_plan_for(*shape, tg.TG_C_BF16, None, 152)
        assert st1 == st2 == tg.TG_OK
        assert (p1.mma, p1.tile_n, p1.stages, p1.grid, p1.sk_iters, p1.split_units) == \
               (p2.mma, p2.tile_n, p2.stages, p2.grid, p2.sk_iters, p2.split_units)
    # the automatic ring depth follows the k-loop: 6 from 32 k-blocks on, else 5
    assert tg.tg_gemm_plan_for(8192, 8192, 8192, tg.TG_C_BF16, None, 152)[1].stages == 6
    assert tg.tg_gemm_plan_for(16384, 4096, 1024, tg.TG_C_BF16, None, 152)[1].stages == 5
    assert tg.tg_gemm_plan_for(8192, 8192, 8192, tg.TG_C_BF16, tg.make_config(stages=4), 152)[1].stages == 4
    assert c.timeout_ns == 1_000_000_000


FAKE = 0x10000  # 16-byte-aligned non-null address; never dereferenced by these tests


def tensor(base=FAKE, dtype=tg.TG_DTYPE_BF16, inner=8200, outer=4100, stride=None, rank=2):
    stride = inner * 2 if stride is None else stride
    return tg.make_tensor2d(base, dtype, inner, outer, stride, rank)


@pytest.mark.parametrize("case,want", [
    (dict(), tg.TG_OK),
    (dict(rank=0), tg.TG_ERR_INVALID_VALUE),
    (dict(rank=6), tg.TG_ERR_INVALID_VALUE),
    (dict(rank=3), tg.TG_ERR_UNSUPPORTED),
    (dict(dtype=9), tg.TG_ERR_INVALID_VALUE),
    (dict(inner=0), tg.TG_ERR_INVALID_VALUE),
    (dict(outer=(1 << 32) + 1), tg.TG_ERR_INVALID_VALUE),
    (dict(base=0), tg.TG_ERR_INVALID_VALUE),
    (dict(base=FAKE + 8), tg.TG_ERR_MISALIGNED),
    (dict(stride=8200 * 2 + 8), tg.TG_ERR_MISALIGNED),
    (dict(stride=8200 * 2 - 16), tg.TG_ERR_INVALID_VALUE),
    (dict(stride=1 << 40), tg.TG_ERR_INVALID_VALUE),
])
def test_tensor_rules(case, want):
    assert tg.tma_validate(tensor(**case), tg.make_box(64, 128), tg.TG_SWZ_128B) == want


@pytest.mark.parametrize("inner,outer,swz,want", [
    (64, 128, tg.TG_SWZ_128B, tg.TG_OK),
    (65, 128, tg.TG_SWZ_128B, tg.TG_ERR_INVALID_VALUE),   # 130 B > 128-byte span
    (32, 128, tg.TG_SWZ_64B, tg.TG_OK),
    (64, 128, tg.TG_SWZ_64B, tg.TG_ERR_INVALID_VALUE),    # 128 B > 64-byte span
    (16, 128, tg.TG_SWZ_32B, tg.TG_OK),
    (32, 128, tg.TG_SWZ_32B, tg.TG_ERR_INVALID_VALUE),    # 64 B > 32-byte span
    (8, 128, tg.TG_SWZ_32B, tg.TG_OK),                    # 16 B <= span
    (4, 128, tg.TG_SWZ_NONE, tg.TG_ERR_MISALIGNED),       # 8 B not a multiple of 16
    (256, 256, tg.TG_SWZ_NONE, tg.TG_OK),
    (257, 1, tg.TG_SWZ_NONE, tg.TG_ERR_INVALID_VALUE),
    (8, 0, tg.TG_SWZ_NONE, tg.TG_ERR_INVALID_VALUE),
    (8, 257, tg.TG_SWZ_NONE, tg.TG_ERR_INVALID_VALUE),
    (64, 128, 4, tg.TG_ERR_INVALID_VALUE),
])
def test_box_rules(inner, outer, swz, want):
    assert tg.tma_validate(tensor(), tg.make_box(inner, outer), swz) == want


def test_validate_null_arguments():
    assert tg.tma_validate(None, tg.make_box(64, 128), 0) == tg.TG_ERR_INVALID_VALUE
    assert tg.tma_validate(tensor(), None, 0) == tg.TG_ERR_INVALID_VALUE


def test_image_bytes_of_copy_configs():
    for w, want in [(64, 69_746_688), (32, 69_476_352), (16, 69_341_184)]:
        assert tg.tma_tile_copy_image_bytes(tensor(), tg.make_box(w, 128)) == want
        assert tg.image_bytes(4100, 8200, 2, w, 128) == want


def copy_err(**kw):
    t = kw.pop("t", tensor())
    box = kw.pop("box", tg.make_box(64, 128))
    swz = kw.pop("swz", tg.TG_SWZ_128B)
    oob = kw.pop("oob", tg.TG_OOB_ZERO)
    out = kw.pop("out", FAKE)
    nbytes = kw.pop("nbytes", 69_746_688)
    return tg.tma_tile_copy(t, box, swz, oob, out, nbytes, None)


def test_copy_host_rules_before_any_launch():
    assert copy_err(out=0) == tg.TG_ERR_INVALID_VALUE
    assert copy_err(out=FAKE + 4) == tg.TG_ERR_MISALIGNED
    assert copy_err(nbytes=69_746_687) == tg.TG_ERR_BUFFER_TOO_SMALL
    assert copy_err(oob=5) == tg.TG_ERR_INVALID_VALUE
    assert copy_err(t=tensor(dtype=tg.TG_DTYPE_U8, stride=8208), oob=tg.TG_OOB_NAN,
                    box=tg.make_box(128, 128)) == tg.TG_ERR_INVALID_VALUE
    # NONE swizzle, 256 x 256 fp32 box = 256 KiB: above the 64 KiB stage limit
    assert copy_err(t=tensor(dtype=tg.TG_DTYPE_F32, stride=8200 * 4), swz=tg.TG_SWZ_NONE,
                    box=tg.make_box(256, 256), nbytes=1 << 40) == tg.TG_ERR_UNSUPPORTED
    # swizzled 3-row box of 32 bytes: 96 bytes, not a multiple of 128
    assert copy_err(box=tg.make_box(16, 3), swz=tg.TG_SWZ_32B,
                    nbytes=1 << 40) == tg.TG_ERR_UNSUPPORTED
    # swizzled boxes narrower than the span are valid descriptors but not provided here
    for w, swz in [(32, tg.TG_SWZ_128B), (8, tg.TG_SWZ_128B), (16, tg.TG_SWZ_64B),
                   (8, tg.TG_SWZ_32B)]:
        assert tg.tma_validate(tensor(), tg.make_box(w, 128), swz) == tg.TG_OK
        assert copy_err(box=tg.make_box(w, 128), swz=swz, nbytes=1 << 40) == tg.TG_ERR_UNSUPPORTED


def test_copy_config_rules():
    for stages, blocks, order, l2p in [(1, 0, 0, 0), (17, 0, 0, 0), (4, 33, 0, 0), (4, 0, 3, 0),
                                       (4, 0, 0, 5)]:
        cfg = tg.tg_copy_config()
        cfg.stages, cfg.blocks_per_sm, cfg.order, cfg.l2_promotion = stages, blocks, order, l2p
        assert tg.tma_tile_copy_ex(tensor(), tg.make_box(64, 128), tg.TG_SWZ_128B, tg.TG_OOB_ZERO,
                                   FAKE, 69_746_688, cfg, None) == tg.TG_ERR_INVALID_VALUE


def gemm_err(M=256, N=256, K=256, A=FAKE, lda=None, B=FAKE, ldb=None, C=FAKE, ldc=None,
             layout=tg.TG_C_F32, cfg=None):
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return tg.gemm_bf16_ex(M, N, K, A, lda, B, ldb, C, ldc, 1.0, 0.0, layout, cfg, None)


def test_gemm_host_rules_before_any_launch():
    assert gemm_err(M=-1) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(K=1 << 31) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(layout=1 << 7) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(layout=7 << 4) == tg.TG_ERR_INVALID_VALUE      # no input type 7
    # MX types (5, 6) carry block scales: gemm_mx only
    assert gemm_err(layout=tg.TG_IN_MXE4M3) == tg.TG_ERR_UNSUPPORTED
    assert gemm_err(layout=tg.TG_IN_MXE5M2) == tg.TG_ERR_UNSUPPORTED
    assert gemm_err(layout=3 << 2) == tg.TG_ERR_INVALID_VALUE      # no C type 3
    # 8-bit operands: K-major only; rows of 16-byte multiples are 16 elements
    for t in (tg.TG_IN_E4M3, tg.TG_IN_E5M2):
        assert gemm_err(layout=t | tg.TG_LAYOUT_A_MN_MAJOR) == tg.TG_ERR_UNSUPPORTED
        assert gemm_err(layout=t | tg.TG_LAYOUT_B_MN_MAJOR) == tg.TG_ERR_UNSUPPORTED
        assert gemm_err(K=264, layout=t) == tg.TG_ERR_MISALIGNED   # 264-byte rows
        assert gemm_err(K=264, lda=272, ldb=272, layout=t) != tg.TG_ERR_MISALIGNED
        assert gemm_err(K=264, lda=272, ldb=272, A=FAKE + 8, layout=t) == tg.TG_ERR_MISALIGNED
    # tf32: K-major only; rows of 16-byte multiples are 4 elements
    t = tg.TG_IN_TF32
    assert gemm_err(layout=t | tg.TG_LAYOUT_A_MN_MAJOR) == tg.TG_ERR_UNSUPPORTED
    assert gemm_err(layout=t | tg.TG_LAYOUT_B_MN_MAJOR) == tg.TG_ERR_UNSUPPORTED
    assert gemm_err(K=258, lda=258, ldb=260, layout=t) == tg.TG_ERR_MISALIGNED   # 1032-byte rows
    assert gemm_err(K=258, lda=260, ldb=260, layout=t) != tg.TG_ERR_MISALIGNED
    assert gemm_err(ldc=260, layout=tg.TG_C_F16) == tg.TG_ERR_MISALIGNED  # 520-byte rows
    # M-major A needs lda >= M, N-major B needs ldb >= N
    assert gemm_err(M=512, lda=256, layout=tg.TG_LAYOUT_A_MN_MAJOR) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(N=512, ldb=256, ldc=512, layout=tg.TG_LAYOUT_B_MN_MAJOR) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(M=512, lda=516, layout=tg.TG_LAYOUT_A_MN_MAJOR) == tg.TG_ERR_MISALIGNED
    assert gemm_err(M=0, A=0, B=0, C=0) == tg.TG_OK          # nothing to do
    assert gemm_err(N=0, A=0, B=0, C=0) == tg.TG_OK
    assert gemm_err(lda=255) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(ldb=100) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(ldc=255) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(A=0) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(C=0) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(A=FAKE + 2) == tg.TG_ERR_MISALIGNED
    assert gemm_err(B=FAKE + 8) == tg.TG_ERR_MISALIGNED
    assert gemm_err(C=FAKE + 4) == tg.TG_ERR_MISALIGNED
    assert gemm_err(lda=260) == tg.TG_ERR_MISALIGNED        # 520 bytes
    assert gemm_err(ldb=257) == tg.TG_ERR_MISALIGNED
    assert gemm_err(ldc=258) == tg.TG_ERR_MISALIGNED         # 1032 bytes (fp32)
    assert gemm_err(ldc=260, layout=tg.TG_C_BF16) == tg.TG_ERR_MISALIGNED  # 520 bytes
    # ragged workload's strides are legal: lda = ldb = 2056 -> 4112 B, ldc = 5000 bf16
    assert gemm_err(M=3000, N=5000, K=2056, layout=tg.TG_C_BF16, ldc=5000) in (
        tg.TG_OK, tg.TG_ERR_CUDA, tg.TG_ERR_UNSUPPORTED)


@pytest.mark.parametrize("field,value", [("stages", 1), ("stages", 7), ("cluster", 3),
                                         ("tile_n", 64), ("tile_n", 192), ("flags", 0x10), ("mma", 4),
                                         ("schedule", 4), ("epi_bufs", 3), ("reserved", 1)])
def test_gemm_config_rules(field, value):
    cfg = tg.make_config(**{field: value})
    assert gemm_err(cfg=cfg) == tg.TG_ERR_INVALID_VALUE


def test_dynamic_schedule_plan_and_rules():
    # one cluster per unit, every unit whole; a cap on the grid contradicts it
    assert gemm_err(cfg=tg.make_config(schedule=3, max_ctas=8)) == tg.TG_ERR_INVALID_VALUE
    for mma, cluster, units in [(2, 2, 1024), (1, 1, 2048), (1, 2, 1024)]:
        cfg = tg.make_config(schedule=3, mma=mma, cluster=cluster, tile_n=256)
        st, plan = tg.tg_gemm_plan_for(8192, 8192, 8192, tg.TG_C_BF16, cfg, 148)
        assert st == tg.TG_OK
        assert (plan.dp_units, plan.sk_iters, plan.grid) == (units, 0, units * cluster)


def test_pair_mma_needs_a_cluster_of_two():
    assert gemm_err(cfg=tg.make_config(mma=2, cluster=1)) == tg.TG_ERR_INVALID_VALUE
    st, plan = tg.tg_gemm_plan_for(8192, 8192, 8192, tg.TG_C_BF16, tg.make_config(mma=2), 148)
    assert st == tg.TG_OK
    assert (plan.mma, plan.cluster, plan.tile_m, plan.tile_n) == (2, 2, 256, 256)
    assert plan.stage_bytes == (128 + 128) * 64 * 2    # A rows + half of the B tile
    st, plan = tg.tg_gemm_plan_for(8192, 8192, 8192, tg.TG_C_BF16,
                                   tg.make_config(mma=2, stages=6), 148)
    assert st == tg.TG_OK and plan.smem_bytes <= 232448


def test_timeout_hook_is_accepted_by_every_kernel():
    # the hook (the first cluster's producers issue nothing) is a legal flag for the
    # per-CTA kernel, its multicast variant and the CTA pair: planning accepts all three
    for kw in ({"mma": 1}, {"mma": 1, "cluster": 2}, {"mma": 2}, {}):
        cfg = tg.make_config(flags=tg.TG_GEMM_FLAG_TEST_SKIP_FIRST_LOAD, **kw)
        st, plan = tg.tg_gemm_plan_for(256, 256, 256, tg.TG_C_F32, cfg, 148)
        assert st == tg.TG_OK, kw
    cfg = tg.make_config(flags=tg.TG_GEMM_FLAG_TEST_SKIP_FIRST_LOAD | 0x4)
    assert gemm_err(cfg=cfg) == tg.TG_ERR_INVALID_VALUE   # unknown flag bits


def test_k_zero_accepts_null_operands_until_the_device_step():
    st = gemm_err(K=0, A=0, B=0, lda=0, ldb=0)
    assert st in (tg.TG_OK, tg.TG_ERR_CUDA, tg.TG_ERR_UNSUPPORTED)


@pytest.mark.parametrize("M,N,K,tile_n,cluster,want_tiles,want_grid", [
    (8192, 8192, 8192, 256, 1, (64, 32, 128), 148),
    (8192, 8192, 8192, 256, 2, (64, 32, 128), 148),
    (256, 256, 256, 256, 1, (2, 1, 4), 2),
    (3000, 5000, 2056, 256, 1, (24, 20, 33), 148),
    (1024, 4096, 16384, 256, 1, (8, 16, 256), 128),
    (1024, 4096, 16384, 128, 2, (8, 32, 256), 148),
    (130, 100, 1, 128, 2, (2, 1, 1), 2),
])
def test_plan(M, N, K, tile_n, cluster, want_tiles, want_grid):
    cfg = tg.make_config(tile_n=tile_n, cluster=cluster, stages=4 if tile_n == 256 else 6,
                         schedule=1)
    st, plan = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_BF16, cfg, 148)
    assert st == tg.TG_OK
    assert (plan.tiles_m, plan.tiles_n, plan.k_blocks) == want_tiles
    assert plan.grid == want_grid
    assert plan.smem_bytes <= 232448
    b_rows = tile_n // 2 if plan.mma == 2 else tile_n   # a CTA pair splits the B tile
    assert plan.stage_bytes == (128 + b_rows) * 64 * 2
    assert plan.mma == (2 if cluster == 2 else 1)


@pytest.mark.parametrize("M,N,K,want_dp,want_sk", [
    # 3072 x 4096 x 4096, CTA pairs on 148 SMs: 192 pair tiles over 74 clusters (2.59
    # waves) -> one whole wave, the remaining 118 tiles (64 k-blocks each) split over all
    # clusters
    (3072, 4096, 4096, 74, 118 * 64),
    # 4096^3 on 148 SMs: three whole waves and 34 tiles (at most half a wave) -> the
    # split tail, not stream-K
    (4096, 4096, 4096, 256, 0),
    # dW: 64 pair tiles < 74 clusters -> data-parallel (auto needs one full wave)
    (1024, 4096, 16384, 64, 0),
    # 8192^3: 1024 tiles, 13.8 waves, efficiency 0.98 -> data-parallel
    (8192, 8192, 8192, 1024, 0),
    # 256^3: data-parallel; the automatic width is 224 (a 224-wide and a 32-wide unit on
    # two pairs finish sooner than one 256-wide unit)
    (256, 256, 256, 2, 0),
])
def test_stream_k_plan(M, N, K, want_dp, want_sk):
    st, plan = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_BF16, None, 148)
    assert st == tg.TG_OK
    assert (plan.dp_units, plan.sk_iters) == (want_dp, want_sk)
    if want_sk:
        assert plan.grid == 148               # every cluster takes a share
        assert plan.sk_iters >= plan.grid // 2
    st, dp = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_BF16, tg.make_config(schedule=1), 148)
    assert dp.sk_iters == 0
    st, sk = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_BF16, tg.make_config(schedule=2), 148)
    assert sk.sk_iters >= plan.sk_iters
    if M == 1024:   # forced: every tile split, 256 k-blocks each
        assert (sk.dp_units, sk.sk_iters) == (0, 64 * 256)


@pytest.mark.parametrize("M,N,K,cfg,sms,want_split,want_grid", [
    # 8192^3 on 152 SMs: 1024 pair tiles on 76 clusters leave 36 for a last wave -> split
    (8192, 8192, 8192, {}, 152, 36, 152),
    # the same on 148 SMs: 62 left on 74 clusters (more than half) -> whole tiles
    (8192, 8192, 8192, {}, 148, 0, 148),
    (8192, 8192, 8192, {"flags": tg.TG_GEMM_FLAG_NO_SPLIT_TAIL}, 152, 0, 152),
    # FFN up: 64 x 16 units, like 8192^3
    (16384, 4096, 1024, {}, 152, 36, 152),
    # fewer units than clusters: every unit split, one cluster per half tile
    (512, 2048, 1024, {"tile_n": 256}, 152, 16, 64),
    (256, 256, 64, {"tile_n": 256}, 152, 1, 4),
    # a capped grid: 10 units on 4 clusters -> 2 whole waves and 2 split units
    (1280, 512, 520, {"tile_n": 256, "max_ctas": 8, "mma": 2}, 152, 2, 8),
    # not with the per-CTA kernel, 224-wide tiles, stream-K, the dynamic schedule
    (8192, 8192, 8192, {"mma": 1}, 152, 0, 152),
    (4096, 4096, 4096, {"tile_n": 224}, 152, 0, 152),
    # FFN down: three whole waves and 28 units -> the split tail is preferred to stream-K
    (16384, 1024, 4096, {}, 152, 28, 152),
    (16384, 1024, 4096, {"schedule": 2}, 152, 0, 152),
    (8192, 8192, 8192, {"schedule": 3}, 152, 0, 2048),
])
def test_split_tail_plan(M, N, K, cfg, sms, want_split, want_grid):
    st, plan = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_BF16, tg.make_config(**cfg), sms)
    assert st == tg.TG_OK
    assert (plan.split_units, plan.grid) == (want_split, want_grid)
    if want_split:
        assert plan.sk_iters == 0


def test_split_tail_not_with_n_major_b():
    st, plan = tg.tg_gemm_plan_for(8192, 8192, 8192, tg.TG_C_BF16 | tg.TG_LAYOUT_B_MN_MAJOR,
                                   None, 152)
    assert st == tg.TG_OK and plan.split_units == 0


def test_split_tail_work_items_cover_every_half_once():
    """Host restatement of the device's data-parallel order: item w of cluster c is
    w = c + j * C; items below split_from are whole units, the rest map to (unit, half)."""
    for units, C in [(1024, 76), (10, 4), (6, 76), (24, 7)]:
        rem = units % C
        split = rem if rem and 2 * rem <= C else 0
        split_from, work = units - split, units + split
        seen = {}
        for c in range(min(work, C)):
            for w in range(c, work, C):
                key = (w, 0) if w < split_from else \
                    (split_from + (w - split_from) // 2, 1 + (w - split_from) % 2)
                seen[key] = seen.get(key, 0) + 1
        want = {(u, 0) for u in range(split_from)} | \
            {(u, h) for u in range(split_from, units) for h in (1, 2)}
        assert set(seen) == want and all(v == 1 for v in seen.values())
        if split:   # the half tiles all fit in one last wave
            assert -(-work // C) == units // C + 1


def test_stream_k_shares_cover_every_iteration_once():
    """Host restatement of the device partition: cluster c owns iterations
    [floor(c*I/C), floor((c+1)*I/C)); a unit split between clusters is finished by the one
    holding its first k-block after adding the partials of the clusters after it."""
    for units, kb, C in [(108, 64, 74), (64, 256, 74), (5, 7, 4), (13, 9, 12)]:
        I = units * kb
        start = lambda c: I * c // C
        seen = [0] * I
        for c in range(C):
            assert start(c + 1) > start(c)           # no empty share
            for it in range(start(c), start(c + 1)):
                seen[it] += 1
        assert all(x == 1 for x in seen)
        for u in range(units):
            first = next(c for c in range(C) if start(c) <= u * kb < start(c + 1))
            last_it = u * kb + kb - 1
            c_last = ((last_it + 1) * C - 1) // I     # the device's formula
            assert start(c_last) <= last_it < start(c_last + 1)
            assert c_last >= first


@pytest.mark.parametrize("in_type", [tg.TG_IN_E4M3, tg.TG_IN_E5M2])
def test_plan_of_8_bit_operands(in_type):
    # the same 128-byte k-block holds 128 elements: half as many k-blocks as bf16
    st, plan = tg.tg_gemm_plan_for(8192, 8192, 8192, tg.TG_C_BF16 | in_type, None, 148)
    assert st == tg.TG_OK
    assert (plan.tile_k, plan.k_blocks, plan.mma) == (128, 64, 2)
    assert plan.stage_bytes == (128 + 128) * 128
    st, plan = tg.tg_gemm_plan_for(4096, 4096, 4100, tg.TG_C_BF16 | in_type,
                                   tg.make_config(mma=1, schedule=1), 148)
    assert st == tg.TG_OK and (plan.tile_k, plan.k_blocks) == (128, 33)


def test_plan_of_tf32_operands():
    # a 128-byte k-block holds 32 binary32 elements
    st, plan = tg.tg_gemm_plan_for(8192, 8192, 8192, tg.TG_C_BF16 | tg.TG_IN_TF32, None, 148)
    assert st == tg.TG_OK
    assert (plan.tile_k, plan.k_blocks, plan.stage_bytes) == (32, 256, (128 + 128) * 128)


def test_plan_rejects_ring_that_does_not_fit():
    st, _ = tg.tg_gemm_plan_for(8192, 8192, 8192, tg.TG_C_BF16,
                                tg.make_config(tile_n=256, stages=5, mma=1), 148)
    assert st == tg.TG_ERR_UNSUPPORTED   # 5 x 48 KiB per-CTA stages do not fit
    st, plan = tg.tg_gemm_plan_for(8192, 8192, 8192, tg.TG_C_BF16,
                                   tg.make_config(tile_n=128, stages=6, mma=1), 148)
    assert st == tg.TG_OK and plan.smem_bytes <= 232448


def test_without_gpu_the_device_step_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert gemm_err() == tg.TG_ERR_CUDA
    assert copy_err() == tg.TG_ERR_CUDA
    assert tg.tg_status_sync(None) == tg.TG_ERR_CUDA


def nd(dims, strides=None, dtype=tg.TG_DTYPE_BF16, base=FAKE):
    es = {tg.TG_DTYPE_U8: 1, tg.TG_DTYPE_BF16: 2, tg.TG_DTYPE_F16: 2, tg.TG_DTYPE_F32: 4}[dtype]
    if strides is None:
        strides, acc = [], dims[0] * es
        for d in dims[1:]:
            strides.append(acc)
            acc *= d
    return tg.make_tensor_nd(base, dtype, dims, strides)


@pytest.mark.parametrize("case,want", [
    (dict(t=nd([64, 8, 4]), b=([64, 4, 2], [1, 1, 2])), tg.TG_OK),
    (dict(t=nd([64, 8, 4, 3, 2]), b=([64, 2, 2, 1, 1], [1, 2, 1, 1, 1])), tg.TG_OK),
    (dict(t=nd([128]), b=([64], [1])), tg.TG_OK),
    (dict(t=nd([64, 8, 4]), b=([64, 4, 2], [2, 1, 1])), tg.TG_ERR_INVALID_VALUE),  # inner stride
    (dict(t=nd([64, 8, 4]), b=([64, 4, 2], [1, 9, 1])), tg.TG_ERR_INVALID_VALUE),  # stride > 8
    (dict(t=nd([64, 8, 4]), b=([64, 4, 2], [1, 0, 1])), tg.TG_ERR_INVALID_VALUE),
    (dict(t=nd([64, 8, 4], [128, 512]), b=([64, 4, 2], [1, 1, 1])), tg.TG_ERR_INVALID_VALUE),  # overlap
    (dict(t=nd([64, 8, 4], [128, 1032]), b=([64, 4, 2], [1, 1, 1])), tg.TG_ERR_MISALIGNED),
    (dict(t=nd([64, 8, 4]), b=([64, 257, 2], [1, 1, 1])), tg.TG_ERR_INVALID_VALUE),
    (dict(t=nd([64, 8, 4, 2, 2]), rank=6, b=([64, 4, 2, 1, 1], [1, 1, 1, 1, 1])),
     tg.TG_ERR_INVALID_VALUE),
    (dict(t=nd([64, 8, 4]), rank=0, b=([64, 4, 2], [1, 1, 1])), tg.TG_ERR_INVALID_VALUE),
])
def test_nd_rules(case, want):
    t = case["t"]
    if "rank" in case:
        t.rank = case["rank"]
    b = tg.make_box_nd(*case["b"])
    assert tg.tma_validate_nd(t, b, tg.TG_SWZ_128B) == want


def test_nd_image_bytes():
    # 3-D bf16 tensor 64 x 10 x 7, box 64 x 4 x 3 with stride 2 on dim 2: L = 64, 4, 2
    t, b = nd([64, 10, 7]), tg.make_box_nd([64, 4, 3], [1, 1, 2])
    assert tg.tma_tile_copy_nd_image_bytes(t, b) == (1 * 3 * 3) * (64 * 4 * 2) * 2
    # rank 2 with unit strides matches the 2-D form
    t2 = tensor()
    assert tg.tma_tile_copy_nd_image_bytes(nd([8200, 4100]), tg.make_box_nd([64, 128])) == \
        tg.tma_tile_copy_image_bytes(t2, tg.make_box(64, 128))


def test_region_copy_host_rules():
    t = tg.make_tensor_nd(FAKE, tg.TG_DTYPE_BF16, [200, 300], [400])
    b = tg.make_box_nd([64, 128])
    ok = tg.tma_validate_region_nd
    assert ok(t, b, [-8, -8], [4, 3], tg.TG_SWZ_128B) == tg.TG_OK
    assert ok(t, b, [-4, 0], [4, 3], tg.TG_SWZ_128B) == tg.TG_ERR_MISALIGNED   # 8 bytes
    assert ok(t, b, [0, -5], [4, 3], tg.TG_SWZ_128B) == tg.TG_OK               # outer: any
    assert ok(t, b, [0, 0], [0, 3], tg.TG_SWZ_128B) == tg.TG_ERR_INVALID_VALUE
    assert ok(t, b, None, [1, 1], tg.TG_SWZ_128B) == tg.TG_ERR_INVALID_VALUE
    assert ok(t, b, [0, 0], None, tg.TG_SWZ_128B) == tg.TG_ERR_INVALID_VALUE
    assert ok(t, b, [0, 2 ** 31 - 128], [1, 2], tg.TG_SWZ_128B) == tg.TG_ERR_INVALID_VALUE
    assert ok(t, b, [0, -2 ** 31], [1, 1], tg.TG_SWZ_128B) == tg.TG_OK
    assert tg.tma_tile_copy_region_nd_image_bytes(t, b, [4, 3]) == 4 * 3 * 64 * 128 * 2
    assert tg.tma_tile_copy_region_nd_image_bytes(t, b, [0, 3]) == 0
    # entries at or beyond the rank are ignored
    assert ok(t, b, [0, 0, 99, 99, 99], [1, 1, 0, 0, 0], tg.TG_SWZ_128B) == tg.TG_OK
    out_small = tg.tma_tile_copy_region_nd(t, b, [0, 0], [4, 3], tg.TG_SWZ_128B, tg.TG_OOB_ZERO,
                                           FAKE, 100, None, None)
    assert out_small == tg.TG_ERR_BUFFER_TOO_SMALL


def test_tensor_rate_probe_rules():
    probe = lambda layout, iters: tg.lib().tg_tensor_rate_probe(layout, iters, None, None)
    assert probe(tg.TG_C_BF16, 16) == tg.TG_ERR_INVALID_VALUE       # only the operand type
    assert probe(5 << 4, 16) == tg.TG_ERR_INVALID_VALUE
    assert probe(tg.TG_IN_BF16, 0) == tg.TG_ERR_INVALID_VALUE
    assert probe(tg.TG_IN_BF16, (1 << 24) + 1) == tg.TG_ERR_INVALID_VALUE
    timed = lambda layout, iters, timing: tg.lib().tg_tensor_rate_probe_timed(layout, iters, None,
                                                                              timing, None)
    assert timed(tg.TG_IN_BF16, 16, None) == tg.TG_ERR_INVALID_VALUE       # needs the buffer
    assert timed(tg.TG_IN_BF16, 16, 0x1004) == tg.TG_ERR_MISALIGNED          # two aligned uint64
    assert timed(tg.TG_C_BF16, 16, 0x1000) == tg.TG_ERR_INVALID_VALUE
    assert timed(tg.TG_IN_BF16, 0, 0x1000) == tg.TG_ERR_INVALID_VALUE


def test_tile_width_224():
    # a pair-tile width only
    assert gemm_err(cfg=tg.make_config(tile_n=224, mma=1)) == tg.TG_ERR_INVALID_VALUE
    st, plan = tg.tg_gemm_plan_for(1024, 4096, 16384, tg.TG_C_BF16, tg.make_config(tile_n=224), 152)
    assert st == tg.TG_OK
    # 4 row pairs x ceil(4096 / 224) = 19 columns = 76 units: one unit per pair of 152 SMs
    assert (plan.tile_m, plan.tile_n, plan.tiles_n, plan.grid) == (256, 224, 19, 152)
    assert plan.stage_bytes == (128 + 112) * 128 and plan.smem_bytes <= 232448


def test_automatic_tile_width():
    # 224 where it fills the waves that 256 leaves poorly filled, on 152 SMs (76 pairs)
    def width(M, N, K=4096, cfg=None):
        st, plan = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_BF16, cfg, 152)
        assert st == tg.TG_OK
        return plan.tile_n
    assert width(1024, 4096, 16384) == 224      # dW: 76 tiles instead of 64
    assert width(4096, 4096) == 224             # four full waves instead of 3.4
    assert width(8192, 8192) == 256             # both fill 96 % of the waves
    assert width(16384, 1024) == 256            # 224 would be worse
    assert width(2048, 2048) == 256
    assert width(3000, 5000, 2056) == 224       # the ragged workload: balance 0.86 vs 0.75
    assert width(16384, 4096, 1024) == 256      # FFN up: equal balance
    assert width(1024, 4096, 16384, tg.make_config(tile_n=256)) == 256   # the caller's choice
    assert width(1024, 4096, 16384, tg.make_config(mma=1)) == 256        # pair tiles only


def test_caller_workspace_rules_on_the_host():
    ws = 0x20000
    # a workspace needs a size and a size needs a workspace; 16-byte alignment
    assert gemm_err(cfg=tg.make_config(workspace=ws)) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(cfg=tg.make_config(workspace_bytes=4096)) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(cfg=tg.make_config(workspace=ws + 8, workspace_bytes=4096)) == \
        tg.TG_ERR_MISALIGNED
    # the plan states the size a stream-K launch needs: the flags (one word per CTA,
    # padded to 256 bytes), then a 128 x tile_n fp32 partial per CTA
    st, plan = tg.tg_gemm_plan_for(1100, 1300, 2000, tg.TG_C_F32, tg.make_config(schedule=2), 148)
    assert st == tg.TG_OK and plan.sk_iters > 0
    flags = -(-plan.grid * 4 // 256) * 256
    assert plan.workspace_bytes == flags + plan.grid * 128 * plan.tile_n * 4
    st, plan = tg.tg_gemm_plan_for(1100, 1300, 2000, tg.TG_C_F32, tg.make_config(schedule=1), 148)
    assert st == tg.TG_OK and plan.sk_iters == 0 and plan.workspace_bytes == 0


def test_last_plan_query():
    st, plan = tg.tg_gemm_last_plan()
    assert st == tg.TG_OK
    assert tg.lib().tg_gemm_last_plan(None) == tg.TG_ERR_INVALID_VALUE


def test_two_pair_cluster_rules_and_plan():
    # mma 3 = two CTA pairs per cluster of four; a cluster of four implies it
    for cfg in (tg.make_config(mma=3), tg.make_config(cluster=4)):
        st, plan = tg.tg_gemm_plan_for(3000, 5000, 2056, tg.TG_C_BF16, cfg, 152)
        assert st == tg.TG_OK and plan.mma == 3 and plan.cluster == 4
        assert plan.tile_m == 256 and plan.grid % 4 == 0 and plan.grid <= 152
        assert plan.stage_bytes == (128 + plan.tile_n // 2) * 128   # A rows + the B half
        assert plan.split_units == 0                               # no split tail
    assert gemm_err(cfg=tg.make_config(mma=3, cluster=2)) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(cfg=tg.make_config(mma=2, cluster=4)) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(cfg=tg.make_config(mma=3, schedule=3)) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(cfg=tg.make_config(mma=4)) == tg.TG_ERR_INVALID_VALUE
    assert gemm_err(cfg=tg.make_config(cluster=3)) == tg.TG_ERR_INVALID_VALUE


def test_plan_follows_the_row_strides():
    # ragged workload: 2056-element rows (4112 bytes) -> the two-pair cluster; rows padded
    # to 2112 elements (4224 bytes, a 128-byte multiple) -> the CTA pair
    L = tg.TG_C_BF16
    st, tight = tg.tg_gemm_plan_for(3000, 5000, 2056, L, None, 152)
    st2, same = tg.tg_gemm_plan_ld(3000, 5000, 2056, 2056, 2056, L, None, 152)
    assert st == st2 == tg.TG_OK and tight.mma == same.mma == 3 and tight.grid == same.grid
    st, padded = tg.tg_gemm_plan_ld(3000, 5000, 2056, 2112, 2112, L, None, 152)
    assert st == tg.TG_OK and padded.mma == 2 and padded.cluster == 2
    st, onlyb = tg.tg_gemm_plan_ld(3000, 5000, 2048, 2048, 2056, L, None, 152)
    assert st == tg.TG_OK and onlyb.mma == 3          # either operand's rows decide
    # kept on the pair: explicit kernel, 8-bit operands, M below two pair tiles
    st, p = tg.tg_gemm_plan_ld(3000, 5000, 2056, 2056, 2056, L, tg.make_config(mma=2), 152)
    assert st == tg.TG_OK and p.mma == 2
    st, p = tg.tg_gemm_plan_ld(3000, 5000, 2064, 2064, 2064, L | tg.TG_IN_E4M3, None, 152)
    assert st == tg.TG_OK and p.mma == 2
    st, p = tg.tg_gemm_plan_ld(500, 5000, 2056, 2056, 2056, L, None, 152)
    assert st == tg.TG_OK and p.mma == 2


def test_driver_symbol_lookup_reports_a_missing_symbol():
    """The lookup that precedes every tensor-map encoding: a name the driver does not
    export gives TG_ERR_NO_DRIVER_SYMBOL (without a driver the runtime cannot be asked at
    all, which is TG_ERR_CUDA)."""
    st = tg.tg_driver_symbol_status("cuTensorMapEncodeTiledThatDoesNotExist")
    assert st in (tg.TG_ERR_NO_DRIVER_SYMBOL, tg.TG_ERR_CUDA)
    assert tg.tg_driver_symbol_status(None) == tg.TG_ERR_INVALID_VALUE


def test_gemm_mx_host_rules():
    S = 0x40000
    L = tg.TG_C_F32 | tg.TG_IN_MXE4M3
    call = lambda **kw: tg.gemm_mx_raw(kw.get("M", 256), 256, kw.get("K", 256), FAKE,
                                       kw.get("lda", 256), kw.get("sa", S), FAKE, 256, S, FAKE,
                                       256, 1.0, 0.0, kw.get("layout", L), kw.get("cfg"))
    assert call(layout=tg.TG_C_F32 | tg.TG_IN_E4M3) == tg.TG_ERR_INVALID_VALUE  # no scales
    assert call(layout=L | tg.TG_LAYOUT_A_MN_MAJOR) == tg.TG_ERR_UNSUPPORTED   # K-major only
    assert call(sa=0) == tg.TG_ERR_INVALID_VALUE
    assert call(sa=S + 4) == tg.TG_ERR_MISALIGNED
    assert call(lda=260) == tg.TG_ERR_MISALIGNED                               # 260-byte rows
    assert call(cfg=tg.make_config(tile_n=224)) == tg.TG_ERR_INVALID_VALUE
    assert call(cfg=tg.make_config(mma=1, tile_n=256)) == tg.TG_ERR_INVALID_VALUE
    assert call(cfg=tg.make_config(mma=2, cluster=4)) == tg.TG_ERR_INVALID_VALUE
    assert call(cfg=tg.make_config(mma=3)) == tg.TG_ERR_INVALID_VALUE
    assert call(cfg=tg.make_config(schedule=2)) == tg.TG_ERR_INVALID_VALUE
    assert call(M=0) == tg.TG_OK
    # scale storage: 512 bytes per (128 rows, 128 elements of K), rounded up
    assert tg.gemm_mx_scale_bytes(300, 200) == 3 * 2 * 512
    assert tg.gemm_mx_scale_bytes(128, 128) == 512 and tg.gemm_mx_scale_bytes(0, 5) == 0
    # default: the CTA pair, 256-wide tiles, 4 stages; each CTA's stage holds its 128 A
    # rows, its 128 B rows, A's scale atom and both B atoms of the tile
    st, plan = tg.tg_gemm_plan_for(8192, 8192, 8192, L, None, 152)
    assert st == tg.TG_OK and (plan.mma, plan.tile_n, plan.stages, plan.cluster) == (2, 256, 4, 2)
    assert plan.stage_bytes == (128 + 128) * 128 + 3 * 512
    assert plan.grid == 152 and plan.split_units == 0 and plan.sk_iters == 0
    st, plan = tg.tg_gemm_plan_for(8192, 8192, 8192, L, tg.make_config(mma=1), 152)
    assert st == tg.TG_OK and (plan.mma, plan.tile_n, plan.stages, plan.cluster) == (1, 128, 5, 1)
    assert plan.stage_bytes == 128 * 128 * 2 + 2 * 512
    # six pair stages do not fit next to the epilogue's staging buffers
    st, _ = tg.tg_gemm_plan_for(8192, 8192, 8192, L, tg.make_config(stages=6), 152)
    assert st == tg.TG_ERR_UNSUPPORTED


@pytest.mark.parametrize("M,N,want", [
    # 256-wide pair tiles on 76 clusters (152 SMs), K = 4096 (64 k-blocks)
    (16384, 1024, "split"),   # 3 full waves + 28 units (at most half a wave): split tail
    (8192, 2560, "split"),    # 4 full waves + 16
    (2560, 4096, "sk"),       # 2 full waves + 8: fewer than three waves before the tail
    (12288, 3072, "sk"),      # 7 full waves + 44: more than half a wave left
])
def test_auto_prefers_split_tail_after_three_waves(M, N, want):
    st, plan = tg.tg_gemm_plan_for(M, N, 4096, tg.TG_C_BF16, tg.make_config(tile_n=256), 152)
    assert st == tg.TG_OK
    units = -(-M // 256) * -(-N // 256)
    if want == "split":
        assert plan.sk_iters == 0 and plan.split_units == units % 76 and plan.dp_units == units
    else:
        assert plan.split_units == 0 and plan.sk_iters > 0
    # an explicit stream-K schedule is never replaced
    st, sk = tg.tg_gemm_plan_for(M, N, 4096, tg.TG_C_BF16, tg.make_config(tile_n=256, schedule=2),
                                 152)
    assert st == tg.TG_OK and sk.sk_iters > 0 and sk.split_units == 0
