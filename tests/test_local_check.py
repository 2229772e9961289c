"""The parity tests' comparison (gdn_testutil.compare) must catch damage that a
whole-tensor relative L2 misses: one wrong (b, t, h) row of o in a tensor the
size of the B4 T2048 H6 training workload, one bad chunk of a gradient, one bad
stream of a state.  CPU only: the mistakes are planted in copies of a reference
tensor, never in the GPU path."""
import numpy as np
import pytest

from gdn_testutil import TOL, compare, rel_l2


def _noisy(ref, rel, rng):
    return ref + rel * np.abs(ref).mean() * rng.standard_normal(ref.shape)


def test_one_wrong_row_of_o_passes_globally_fails_locally():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((4, 2048, 6, 128))
    got = _noisy(ref, 3e-3, rng)
    got[2, 1000, 3, :] = -got[2, 1000, 3, :]  # one row flipped
    assert rel_l2(got, ref) <= TOL["bf16"]["out"]  # the whole-tensor norm hides it
    with pytest.raises(AssertionError, match=r"o: block \(b, chunk, h\)=\(2, 15, 3\)"):
        compare(dict(o=got), dict(o=ref), "bf16")


def test_accurate_tensors_pass():
    rng = np.random.default_rng(1)
    ref = dict(o=rng.standard_normal((2, 300, 3, 64)), dq=rng.standard_normal((2, 300, 3, 32)),
               dalpha=rng.standard_normal((2, 300, 3)), final_state=rng.standard_normal((2, 3, 64, 32)))
    got = {n: _noisy(r, 3e-3, rng) for n, r in ref.items()}
    errs = compare(got, ref, "bf16")
    assert set(errs) == set(ref)


def test_bad_tail_chunk_and_bad_stream_are_named():
    rng = np.random.default_rng(2)
    ref = rng.standard_normal((1, 200, 2, 32))
    got = _noisy(ref, 1e-3, rng)
    got[0, 192:, 1] *= 1.2  # the ragged tail chunk (tokens 192-199) of head 1
    assert rel_l2(got, ref) <= TOL["bf16"]["grad"]
    with pytest.raises(AssertionError, match=r"dk: block \(b, chunk, h\)=\(0, 3, 1\)"):
        compare(dict(dk=got), dict(dk=ref), "bf16")
    s_ref = rng.standard_normal((8, 6, 16, 16))
    s_got = _noisy(s_ref, 1e-3, rng)
    s_got[5, 4] *= 1.1
    assert rel_l2(s_got, s_ref) <= TOL["bf16"]["out"]
    with pytest.raises(AssertionError, match=r"final_state: block \(b, h\)=\(5, 4\)"):
        compare(dict(final_state=s_got), dict(final_state=s_ref), "bf16")


def test_chunk_size_sets_the_token_blocks():
    rng = np.random.default_rng(3)
    ref = rng.standard_normal((1, 256, 1, 16))
    got = ref.copy()
    got[0, 40:48] *= 1.1  # half of a 16-token chunk, an eighth of a 64-token one
    compare(dict(o=got), dict(o=ref), "bf16", chunk=64)
    with pytest.raises(AssertionError, match=r"\(0, 2, 0\)"):
        compare(dict(o=got), dict(o=ref), "bf16", chunk=16)
