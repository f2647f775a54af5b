"""Pins for the layout oracle (document ids from lengths, document positions,
the position validator, the needed key/value range), checked against values
derived by hand from the pages' definitions and against brute force.

Pages: "nemo_automodel.components.models.glm5_next.cp" (doc_ids_from_seq_lens),
"nemo_automodel.components.models.inkling2.context_parallel"
(unpack_row_layout, validate_document_positions) and
"nemo_automodel.components.distributed.blockdiag_cp" (cp_blockdiag_sdpa, the
needed-only K/V exchange).
"""
import numpy as np
import pytest

from oracle import layout as lay


# ----------------------------------------------------------- doc ids from lengths

def test_doc_ids_from_seq_lens_hand_example():
    # lengths of the tiny workload's documents: 37, 100, 1, 64, 54 fill 256 tokens
    ids = lay.doc_ids_from_seq_lens([[37, 100, 1, 64, 54]], 256)
    want = np.array([1] * 37 + [2] * 100 + [3] * 1 + [4] * 64 + [5] * 54, np.int32)
    np.testing.assert_array_equal(ids[0], want)


def test_doc_ids_from_seq_lens_padding_entries_and_tail():
    ids = lay.doc_ids_from_seq_lens([[3, 2, -1000, -1000], [1, -1000, 2, -1000]], 8)
    np.testing.assert_array_equal(ids[0], [1, 1, 1, 2, 2, 0, 0, 0])
    # a padding entry in the middle takes no number
    np.testing.assert_array_equal(ids[1], [1, 2, 2, 0, 0, 0, 0, 0])


def test_doc_ids_from_seq_lens_zero_length_document_takes_a_number():
    ids = lay.doc_ids_from_seq_lens([[2, 0, 3]], 6)
    np.testing.assert_array_equal(ids[0], [1, 1, 3, 3, 3, 0])


def test_doc_ids_from_seq_lens_custom_padding_value():
    ids = lay.doc_ids_from_seq_lens([[2, -1, 1]], 4, padding_value=-1)
    np.testing.assert_array_equal(ids[0], [1, 1, 2, 0])


@pytest.mark.parametrize("lens,S", [([[3, -2]], 8), ([[5, 4]], 8)])
def test_doc_ids_from_seq_lens_rejects(lens, S):
    with pytest.raises(ValueError):
        lay.doc_ids_from_seq_lens(lens, S)


# ----------------------------------------------------------- positions from ids

def test_positions_hand_example():
    pos, keep = lay.position_ids_from_doc_ids([[1, 1, 1, 0, 0, 2, 2, 3]])
    np.testing.assert_array_equal(pos[0], [0, 1, 2, 0, 0, 0, 1, 0])
    np.testing.assert_array_equal(keep[0], [1, 1, 1, 0, 0, 1, 1, 1])


def test_positions_restart_after_a_gap_in_a_repeated_id():
    # the second run of id 1 is another segment: it restarts at 0
    pos, keep = lay.position_ids_from_doc_ids([[1, 1, 0, 1, 1]])
    np.testing.assert_array_equal(pos[0], [0, 1, 0, 0, 1])


# ----------------------------------------------------------- validator

@pytest.mark.parametrize("keep,pos,bad", [
    ([1, 1, 1, 1, 1], [5, 6, 7, 0, 1], -1),      # shard starts inside a document
    ([0, 0, 1, 1], [9, 9, 4, 5], -1),            # after left padding, any start offset
    ([1, 1, 1], [0, 1, 3], 2),                    # not a unit step
    ([1, 1, 0, 1], [0, 1, 0, 2], 3),              # a gap cannot resume the old document
    ([1, 1, 0, 1], [0, 1, 0, 0], -1),             # after a gap a new document starts at 0
    ([1, 1], [-1, 0], 0),                         # negative start
    ([1, 1, 1], [3, 3, 4], 1),                    # repeated position
    ([0, 0, 0], [7, -5, 2], -1),                  # nothing valid: nothing to check
])
def test_validator_hand_cases(keep, pos, bad):
    assert lay.validate_document_positions([keep], [pos])[0] == bad


def test_validator_accepts_positions_made_from_ids():
    rng = np.random.default_rng(3)
    for _ in range(50):
        S = int(rng.integers(1, 40))
        ids = rng.integers(0, 4, size=(2, S))
        pos, keep = lay.position_ids_from_doc_ids(ids)
        np.testing.assert_array_equal(lay.validate_document_positions(keep, pos), [-1, -1])


def test_validator_rejects_a_single_perturbation():
    rng = np.random.default_rng(4)
    for _ in range(50):
        ids = np.repeat(rng.integers(1, 5, size=6), rng.integers(1, 5, size=6))[None, :]
        pos, keep = lay.position_ids_from_doc_ids(ids)
        p = int(rng.integers(1, ids.shape[1]))  # every row holds >= 6 tokens
        pos2 = pos.copy()
        pos2[0, p] = pos[0, p - 1] + 3  # neither 0 nor the predecessor's position + 1
        assert lay.validate_document_positions(keep, pos2)[0] == p


# ----------------------------------------------------------- needed K/V range

def _brute_needed(ids, s0, L):
    """Union of the dense per-document causal masks of the local queries."""
    S = ids.size
    need = np.zeros(S, bool)
    for t in range(s0, s0 + L):
        if ids[t] == 0:
            continue
        for j in range(t + 1):
            if all(ids[x] == ids[t] for x in range(j, t + 1)):
                need[j] = True
    idx = np.nonzero(need)[0]
    return (int(idx[0]), int(idx[-1]) + 1) if idx.size else None


def test_needed_range_matches_brute_force():
    rng = np.random.default_rng(5)
    for _ in range(60):
        S = int(rng.integers(2, 48))
        ids = np.repeat(rng.integers(0, 4, size=S), 1)[:S]
        ids = np.sort(rng.integers(0, 5, size=S)) if rng.random() < 0.5 else ids
        L = int(rng.integers(1, S + 1))
        s0 = int(rng.integers(0, S - L + 1))
        got = lay.kv_needed_range(ids, s0, L)
        want = _brute_needed(ids, s0, L)
        if want is None:
            assert got == (s0, s0)
        else:
            assert got == want


def test_needed_range_hand_example_and_shards():
    ids = np.array([1] * 37 + [2] * 100 + [3] * 1 + [4] * 64 + [5] * 54, np.int32)
    # queries 100..149: the first lies in document 2 (starting at 37)
    lo, hi = lay.kv_needed_range(ids, 100, 50)
    assert (lo, hi) == (37, 150)
    np.testing.assert_array_equal(lay.kv_rows_per_shard(lo, hi, 256, 50),
                                  [13, 50, 50, 0, 0, 0])
    # the last 20 positions of a row whose tail is padding
    ids2 = np.array([1] * 10 + [0] * 10, np.int32)
    assert lay.kv_needed_range(ids2, 10, 10) == (10, 10)
