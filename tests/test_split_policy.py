"""Host-side choice between ft_cache_step and ft_cache_step_split (no GPU)."""
import expert_cache_streaming_fp32_b300 as ft


def test_split_policy_per_format_and_batch():
    # BF16 decode: the split form from 64 assignments (T=8 at top-8) up to the large-batch tiling
    assert not ft.split_pays(1, 8, ft.FT_W_BF16)
    assert not ft.split_pays(4, 8, ft.FT_W_BF16)
    assert ft.split_pays(8, 8, ft.FT_W_BF16)
    assert ft.split_pays(64, 8, ft.FT_W_BF16)
    assert ft.split_pays(255, 8, ft.FT_W_BF16)
    assert not ft.split_pays(256, 8, ft.FT_W_BF16)          # 2048 assignments: prefill tiling
    assert not ft.split_pays(8192, 8, ft.FT_W_BF16)
    # FP4 decode: from one token
    for w in (ft.FT_W_NVFP4, ft.FT_W_MXFP4):
        assert ft.split_pays(1, 6, w) and ft.split_pays(1, 8, w)
        assert not ft.split_pays(8192, 8, w)
    # an explicit threshold overrides the table
    assert ft.split_pays(1, 8, ft.FT_W_BF16, min_assignments=8)
    assert not ft.split_pays(1, 8, ft.FT_W_NVFP4, min_assignments=16)
    assert ft.SPLIT_MAX_ASSIGNMENTS == ft.FT_TC_WIDE_ASSIGNMENTS == 2048
