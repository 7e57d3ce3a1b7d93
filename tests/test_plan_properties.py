"""Properties of the host planner (no GPU): for any sizes, layouts and tuning knobs that
tg_gemm_plan_for accepts, the launch it describes is self-consistent.  Every tile of the
output belongs to exactly one work item, the grid fits the SMs, and the split tail and
stream-K never combine."""
import pytest

from tma_pipelined_tensor_gb300 import tg

hyp = pytest.importorskip("hypothesis")
st = hyp.strategies

LAYOUTS = [tg.TG_C_BF16, tg.TG_C_F32, tg.TG_C_F16, tg.TG_C_BF16 | tg.TG_IN_E4M3,
           tg.TG_C_BF16 | tg.TG_IN_TF32, tg.TG_C_BF16 | tg.TG_LAYOUT_A_MN_MAJOR,
           tg.TG_C_BF16 | tg.TG_LAYOUT_B_MN_MAJOR]


def work_items(units, clusters, split):
    """The data-parallel order of the kernels: item w of cluster c is w = c + j * clusters;
    units [0, units - split) whole, the last `split` units as two half tiles."""
    split_from = units - split
    seen = {}
    for c in range(clusters):
        for w in range(c, units + split, clusters):
            key = (w, 0) if w < split_from else \
                (split_from + (w - split_from) // 2, 1 + (w - split_from) % 2)
            seen[key] = seen.get(key, 0) + 1
    return seen


@hyp.settings(max_examples=300, deadline=None)
@hyp.given(M=st.integers(1, 40000), N=st.integers(1, 40000), K=st.integers(0, 20000),
           layout=st.sampled_from(LAYOUTS), sms=st.sampled_from([148, 152, 132, 16]),
           tile_n=st.sampled_from([0, 128, 224, 256]), mma=st.sampled_from([0, 1, 2]),
           schedule=st.sampled_from([0, 1, 2, 3]), max_ctas=st.sampled_from([0, 8, 30]),
           no_split=st.booleans())
def test_plan_is_consistent(M, N, K, layout, sms, tile_n, mma, schedule, max_ctas, no_split):
    if schedule == 3:
        max_ctas = 0                      # the dynamic schedule needs the whole grid
    if tile_n == 224 and mma == 1:
        tile_n = 0                        # a pair-tile width only
    cfg = tg.make_config(tile_n=tile_n, mma=mma, schedule=schedule, max_ctas=max_ctas,
                         flags=tg.TG_GEMM_FLAG_NO_SPLIT_TAIL if no_split else 0)
    status, plan = tg.tg_gemm_plan_for(M, N, K, layout, cfg, sms)
    if status != tg.TG_OK:
        # only the documented refusals: N-major B with 224-wide tiles, or a ring that
        # does not fit
        assert status == tg.TG_ERR_UNSUPPORTED
        return
    assert plan.smem_bytes <= 232448
    assert plan.grid % plan.cluster == 0
    units = -(-plan.tiles_m // plan.cluster) * plan.tiles_n
    clusters = plan.grid // plan.cluster
    if schedule == 3:
        assert clusters == units          # one cluster per unit
        assert plan.split_units == 0 and plan.sk_iters == 0
        return
    cap = sms // plan.cluster
    if max_ctas:
        cap = min(cap, max(1, max_ctas // plan.cluster))
    assert 1 <= clusters <= cap
    assert not (plan.split_units and plan.sk_iters)
    if plan.sk_iters:
        assert clusters == cap                          # every usable cluster takes a share
        assert plan.sk_iters == (units - plan.dp_units) * plan.k_blocks
        assert plan.sk_iters >= clusters
        return
    assert plan.dp_units == units
    s = plan.split_units
    if s:
        assert no_split is False and plan.mma == 2 and plan.tile_n == 256
        assert not layout & tg.TG_LAYOUT_B_MN_MAJOR
        assert 2 * s <= cap and s == (units % cap if units >= cap else units)
    seen = work_items(units, clusters, s)
    want = {(u, 0) for u in range(units - s)} | \
        {(u, h) for u in range(units - s, units) for h in (1, 2)}
    assert set(seen) == want and all(v == 1 for v in seen.values())
    # the grid never holds an idle cluster
    assert clusters == min(cap, units + s)
