"""CPU-only checks of the host's reader of a pass's published result.

A pass publishes its 18 sums to mapped host memory as 38 tagged 64-bit words
with no fence: each word holds the pass's tag (low 32 bits of its sequence
number, top bit set) above a payload -- the float bits of each sum's hi and
lo halves, then the low 32 bits of the pass's start and publish times.  The
words may land in any order, so the reader must take a result only when
every word names the pass.  These tests drive the library's own reader
(icpnn_probe_read_result) with words built here from that layout."""
import numpy as np
import pytest

import icp_nearest_neighbour_gb300 as nn

N_SLOTS = 18


def tag(seq: int) -> int:
    return ((seq & 0xFFFFFFFF) | 0x80000000) & 0xFFFFFFFF


def pack(seq: int, hi, lo, t0: int, t1: int) -> np.ndarray:
    payload = np.empty(nn.RESULT_WORDS, dtype=np.uint64)
    payload[0:2 * N_SLOTS:2] = np.asarray(hi, dtype=np.float32).view(np.uint32)
    payload[1:2 * N_SLOTS:2] = np.asarray(lo, dtype=np.float32).view(np.uint32)
    payload[2 * N_SLOTS] = t0 & 0xFFFFFFFF
    payload[2 * N_SLOTS + 1] = t1 & 0xFFFFFFFF
    return payload | np.uint64(tag(seq) << 32)


def random_pairs(rng):
    """Float-float pairs as the device leaves them: |lo| at most half an ulp of hi."""
    hi = rng.standard_normal(N_SLOTS).astype(np.float32) * np.float32(1e3)
    ulp = np.spacing(np.abs(hi)).astype(np.float32)
    lo = (rng.uniform(-0.5, 0.5, N_SLOTS).astype(np.float32) * ulp).astype(np.float32)
    return hi, lo


def test_complete_result_decodes_exactly():
    rng = np.random.default_rng(7)
    hi, lo = random_pairs(rng)
    got = nn.probe_read_result(pack(5, hi, lo, 1_000, 38_500), 5)
    assert got is not None
    slots, ms = got
    want = hi.astype(np.float64) + lo.astype(np.float64)  # exact: the pair spans at most 48 bits
    assert np.array_equal(slots, want)
    assert ms == pytest.approx(0.0375, rel=1e-6)


def test_counts_and_large_sums_survive_the_pair_split():
    # a count above float32's 24-bit range and a sum that needs the lo half
    big = 2.0 ** 30 + 3.0
    hi = np.zeros(N_SLOTS, dtype=np.float32)
    lo = np.zeros(N_SLOTS, dtype=np.float32)
    hi[0] = np.float32(big)
    lo[0] = np.float32(big - float(np.float32(big)))
    slots, _ = nn.probe_read_result(pack(9, hi, lo, 0, 0), 9)
    assert slots[0] == big


@pytest.mark.parametrize("position", range(38))
def test_one_word_of_another_pass_keeps_the_result_incomplete(position):
    rng = np.random.default_rng(position)
    hi, lo = random_pairs(rng)
    w = pack(1234, hi, lo, 10, 20)
    stale = pack(1233, hi, lo, 10, 20)  # the previous pass's word at that position
    w[position] = stale[position]
    assert nn.probe_read_result(w, 1234) is None
    assert nn.probe_read_result(w, 1233) is None


def test_zeroed_memory_is_never_a_result():
    w = np.zeros(nn.RESULT_WORDS, dtype=np.uint64)
    for seq in (0, 1, 2 ** 31, 2 ** 32):
        assert nn.probe_read_result(w, seq) is None


def test_pass_time_wraps_modulo_2_to_the_32():
    hi = np.zeros(N_SLOTS, dtype=np.float32)
    lo = np.zeros(N_SLOTS, dtype=np.float32)
    t0 = 2 ** 32 - 1_000   # start just before the low 32 bits wrap
    t1 = 2 ** 32 + 41_000  # publish just after
    _, ms = nn.probe_read_result(pack(3, hi, lo, t0, t1), 3)
    assert ms == pytest.approx(0.042, rel=1e-6)


def test_wrong_length_is_rejected():
    with pytest.raises(nn.IcpnnError) as e:
        nn.probe_read_result(np.zeros(37, dtype=np.uint64), 1)
    assert e.value.status == "INVALID_ARG"
