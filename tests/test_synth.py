"""The seeded input generators (tree_verified_speculative_gb300/synth.py):
shapes, seeding and the stated structure of the inputs, on the CPU."""
import numpy as np

from tree_verified_speculative_gb300 import synth


def test_vocab_subset_is_an_increasing_sample():
    ids = synth.vocab_subset(151936, 65536, seed=3)
    assert ids.dtype == np.int32 and ids.shape == (65536,)
    assert np.all(np.diff(ids) > 0) and ids[0] >= 0 and ids[-1] < 151936
    assert np.array_equal(ids, synth.vocab_subset(151936, 65536, seed=3))
    assert not np.array_equal(ids, synth.vocab_subset(151936, 65536, seed=4))


def test_futures_share_positions_and_stay_in_the_vocabulary():
    rng = np.random.default_rng(1)
    fut = synth.futures(8, 15, 1000, 11, rng)
    assert fut.shape == (8, 15) and fut.min() >= 0 and fut.max() < 1000
    same = np.all(fut == fut[0:1], axis=0)
    assert same.sum() >= 11  # the shared positions (others may agree by chance)
    ids = synth.vocab_subset(1000, 50, seed=2)
    fut2 = synth.futures(8, 15, 1000, 11, np.random.default_rng(1), vocab=ids)
    assert np.isin(fut2, ids).all()
    assert np.all(fut2 == fut2[0:1], axis=0).sum() >= 11


def test_futures_without_a_vocabulary_keep_their_stream():
    """The draft-vocabulary option leaves the default draws unchanged."""
    a = synth.futures(4, 6, 500, 2, np.random.default_rng(9))
    b = synth.futures(4, 6, 500, 2, np.random.default_rng(9), vocab=None)
    assert np.array_equal(a, b)


def test_plant_sites_follow_the_future():
    # a chain tree root -> 5 -> 7 -> 9 and a side node root -> 6
    parent = np.array([-1, 0, 1, 2, 0])
    token = np.array([0, 5, 7, 9, 6])
    depth = np.array([0, 1, 2, 3, 1])
    rows, cols = synth.plant_sites(parent, token, depth, 5, np.array([5, 7, 8, 4]))
    # root plants 5; node 1 (5) plants 7; node 2 (5, 7) plants 8; node 3 is off the future
    assert list(rows) == [0, 1, 2] and list(cols) == [5, 7, 8]
    t = synth.plant(np.zeros((5, 10), np.float32), rows, cols)
    assert t[0, 5] == 10 and t[1, 7] == 10 and t[2, 8] == 10 and t.sum() == 30
