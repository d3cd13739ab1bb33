"""Seeded input generators: determinism, shapes and the drawn distributions."""
import numpy as np
import pytest

from combine_top_histogram_gb300 import workloads as W


def test_configs_match_the_workload_table():
    assert (W.WORKED.P, W.WORKED.Tr, W.WORKED.E, W.WORKED.k, W.WORKED.H) == (4, 2, 8, 2, 128)
    assert (W.DECODE.T, W.DECODE.E, W.DECODE.k, W.DECODE.H, W.DECODE.Na) == (1024, 256, 8, 7168, 8192)
    assert (W.UNIFORM_FP8.T, W.UNIFORM_FP8.E, W.UNIFORM_FP8.Na) == (16384, 64, 32768)
    assert (W.SKEWED.T, W.SKEWED.E, W.SKEWED.H, W.SKEWED.Na) == (32768, 8, 4096, 65536)
    assert (W.PREFILL.T, W.PREFILL.Na, W.PREFILL.cap) == (131072, 1048576, 5120)
    assert W.PREFILL.rows_max == min(W.PREFILL.Na, 256 * 5120) == 1048576


def test_generation_is_deterministic():
    wl = W.UNIFORM_FP8.scaled("t", Tr=16, H=256)
    a, b = W.make_inputs(wl), W.make_inputs(wl)
    assert np.array_equal(a.x, b.x) and np.array_equal(a.ids, b.ids) and np.array_equal(a.w, b.w)
    c = W.make_inputs(wl, seed=99)
    assert not np.array_equal(a.x, c.x)


def test_shapes_and_ranges():
    for name, wl in W.CONFIGS.items():
        small = wl if name == "worked" else wl.scaled("s", Tr=8, H=256)
        inp = W.make_inputs(small)
        assert inp.x.shape == (small.T, small.H) and inp.x.dtype == np.uint16
        if small.routing == "logits":
            assert inp.logits.shape == (small.T, small.E) and inp.ids is None
        else:
            assert inp.ids.shape == (small.T, small.k)
            assert inp.ids.min() >= 0 and inp.ids.max() < small.E
            # distinct experts per token
            assert all(len(set(r)) == small.k for r in inp.ids.tolist())
            np.testing.assert_allclose(inp.w.sum(axis=1), 1.0, rtol=1e-6)
        if small.expert == "scale":
            assert inp.expert_scale.min() >= 0.5 and inp.expert_scale.max() < 1.5


def test_zipf_first_draw_follows_popularity():
    wl = W.SKEWED.scaled("z", Tr=2048, H=8)
    inp = W.make_inputs(wl)
    p = (np.arange(8) + 1.0) ** -1.2
    p /= p.sum()
    freq = np.bincount(inp.ids[:, 0], minlength=8) / wl.T
    sigma = np.sqrt(p * (1 - p) / wl.T)
    assert np.all(np.abs(freq - p) < 5 * sigma)
    # the hottest expert takes the largest share of all assignments
    tot = np.bincount(inp.ids.reshape(-1), minlength=8)
    assert tot.argmax() == 0 and tot[0] > 2.5 * tot.mean()


def test_worked_inputs_are_the_printed_routing():
    inp = W.make_inputs(W.WORKED)
    assert inp.ids.tolist() == W.WORKED_ROUTING.tolist()
    assert np.all(inp.w == np.array([0.6, 0.4], np.float32))


def test_prefill_capacity_formula():
    assert W.prefill_capacity(32 * 4096, 8, 256) == 5120
    assert W.prefill_capacity(10, 3, 7) == 6  # ceil(1.25*30/7) = ceil(5.36)


@pytest.mark.parametrize("frac", [0.0, 0.5, 1.0])
def test_mask_random_slots(frac):
    ids = np.zeros((100, 4), np.int32)
    m = W.mask_random_slots(ids, frac, 3)
    share = (m == -1).mean()
    assert abs(share - frac) < 0.1
