"""The forward's work decomposition on the host (attn_fwd_schedule; no GPU): which walk a
launch takes, and that the walk with the constants the launch writes visits every
sub-unit exactly once, whatever the grid."""
import pytest

import exact_attention_55_gb300 as fa


@pytest.fixture(scope="module")
def sched():
    from exact_attention_55_gb300 import build
    fa.load_library(build.build())
    return fa.attn_fwd_schedule


def _walk(s_info, c):
    """Sub-units CTA c visits: the kernel's rule, restated from the header's contract."""
    s = c * s_info["first"]
    out = []
    while s < s_info["subs"]:
        out.append(s)
        s = s + 1 + (0 if (s + s_info["a"]) % s_info["m"] == 0 else s_info["step"])
    return out


def _visits(s_info):
    seen = []
    for c in range(s_info["grid"]):
        seen += _walk(s_info, c)
    return seen


def test_walk_choice(sched):
    # headline: 4096 pairs balance as pairs (27 rounds), as do causal launches
    assert sched(16, 16, 8192, 128)["walk"] == 0
    assert sched(16, 16, 8192, 128, causal=True)["walk"] == 0
    assert sched(2, 16, 8192, 128, causal=True)["walk"] == 0
    # 512 pairs on 152 SMs: single units (7 rounds against 8 unit-times)
    assert sched(2, 16, 8192, 128)["walk"] == 1
    assert sched(2, 8, 8192, 256)["walk"] == 1
    # windows: rotated rounds
    assert sched(1, 16, 16384, 128, causal=True, window=1024)["walk"] == 2
    assert sched(8, 16, 2048, 128, causal=True, window=1024)["walk"] == 2
    # a window of N - 1 keys or more is walked as its plain mask
    assert sched(32, 16, 512, 128, causal=True, window=1024)["walk"] == 0
    assert sched(32, 16, 512, 128, causal=False, window=511)["walk"] == 1


def test_grid_and_sizes(sched):
    s = sched(16, 16, 8192, 128)
    assert (s["grid"], s["subs"], s["num_qblk"]) == (152, 8192, 32)
    s = sched(2, 8, 8192, 256)          # 128-row units at d = 256
    assert (s["num_qblk"], s["subs"]) == (64, 2 * 16 * 32)
    s = sched(1, 2, 128, 64, sm_count=152)
    assert s["grid"] == 4 and s["subs"] == 4   # single units: one CTA per sub-unit
    s = sched(1, 2, 128, 64, causal=True, sm_count=152)
    assert s["grid"] == 2                      # pairs: one CTA per pair


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 1024), (False, 300)])
@pytest.mark.parametrize("sm_count", [1, 3, 7, 148, 152, 160])
def test_every_sub_unit_once(sched, causal, window, sm_count):
    for B, H, N, d in [(16, 16, 8192, 128), (2, 16, 8192, 128), (1, 3, 1000, 64), (3, 5, 2048, 256),
                       (8, 16, 2048, 128), (1, 1, 1, 128), (7, 2, 640, 64)]:
        s = sched(B, H, N, d, causal=causal, window=window, sm_count=sm_count)
        assert s["grid"] <= sm_count
        seen = _visits(s)
        assert sorted(seen) == list(range(s["subs"])), (B, H, N, d, s)


def test_rotated_rounds_move_each_cta_along_a_head(sched):
    # B8 H16 N2048 d128 under a 1024-key window: 8 units per head, 152 CTAs (a multiple
    # of 8); a plain stride would give each CTA the same position in every round
    s = sched(8, 16, 2048, 128, causal=True, window=1024)
    units_per_head = 2 * ((s["num_qblk"] + 1) // 2)
    for c in range(s["grid"]):
        pos = [u % units_per_head for u in _walk(s, c)]
        assert len(set(pos)) == len(pos)           # a different position every round
        assert all((b - a) % units_per_head == 1 for a, b in zip(pos, pos[1:]))


def test_argument_errors(sched):
    with pytest.raises(fa.AttnError):
        sched(0, 1, 1, 128)
    with pytest.raises(fa.AttnError):
        sched(1, 1, 1, 96)
    with pytest.raises(fa.AttnError):
        sched(1, 1, 1, 128, sm_count=0)
