"""GPU parity of the multi-block staircase (several active blocks per
trajectory; ORL announcement thread, 24vids.com mirror, Insight 3, replays
"irregular trajectories" with the staircase kernel; ORL paper card,
thelatestinai.com, Figure 3 caption): the CUDA path through the C ABI
against the fp64 oracle, every output element, on the same seeded inputs.

Layouts: the two hand-drawn golden layouts scaled to the kernels' tile
sizes; four groups of eight 32-token copies after a 1,024-token prefix (the
copies of later blocks see more of the prefix); a ragged layout (prefix not
a multiple of 128, empty groups, a group that sees nothing of the prefix)
whose backward key tiles need two separate query ranges; and d = 64."""
import pytest
import torch

from diffusion_lm_block_bda_b300 import workloads as W

from _parity import compare_full, gpu_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")


def _golden(scale, which):
    """A layout of tests/golden/masks_multi.txt with every length x scale:
    "two_groups" (B=2, P=6, groups (2, 2), (1, 6)) or
    "ragged_prefix_empty_group" (B=3, P=5, groups (1, 0), (0, 3), (2, 5))."""
    B, P, g = {"two": (2, 6, [(2, 2), (1, 6)]),
               "ragged": (3, 5, [(1, 0), (0, 3), (2, 5)])}[which]
    return W.multi_staircase([P * scale, P * scale], [[(c, v * scale) for c, v in g]] * 2,
                             block_size=B * scale, hq=8, hkv=2)


CASES = {
    "golden_two_groups_x16": lambda: _golden(16, "two"),
    "golden_ragged_x16": lambda: _golden(16, "ragged"),
    "golden_two_groups_x32": lambda: _golden(32, "two"),
    "golden_ragged_x32": lambda: _golden(32, "ragged"),
    # 4 groups x 8 copies of 32 tokens after a 1,024-token prefix, 2 trajectories
    "four_groups_x8": lambda: W.multi_staircase(
        [1024, 1024], [[(8, 256), (8, 512), (8, 768), (8, 1024)]] * 2, block_size=32),
    # ragged: prefix 1000 (not % 128), empty groups, two query ranges per key tile
    "ragged_two_ranges": lambda: W.multi_staircase(
        [1000, 130], [[(3, 0), (2, 640), (0, 700), (1, 1000)], [(0, 5), (4, 130)]],
        block_size=16, hq=8, hkv=2),
    "d64": lambda: W.multi_staircase(
        [300, 64], [[(2, 100), (3, 300)], [(5, 64)]], block_size=32, hq=8, hkv=2, head_dim=64),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_multi_block_staircase_full_oracle(name):
    w = CASES[name]()
    inp = W.make_inputs(w, seed=13)
    got = gpu_run(w, inp)
    compare_full(w, inp, got)
