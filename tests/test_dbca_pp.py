"""The DBCA-PP width assignment (host-side, no GPU): brute force over the
widths against the rule stated in include/agoq.h, closed cases, and the
memory balance it promises."""
import itertools

import pytest

from gradient_quantization_gb300 import agoq

WIDTHS = (4, 5, 6, 8)


def _live(stages, microbatches, s):
    return min(stages - s, microbatches)


@pytest.mark.parametrize("stages", [1, 2, 3, 4, 6, 8, 16])
@pytest.mark.parametrize("microbatches", [1, 2, 4, 8, 32])
@pytest.mark.parametrize("base", WIDTHS)
def test_widths_are_the_largest_within_the_first_stage_footprint(stages, microbatches, base):
    bits = agoq.agoq_dbca_pp_bits(stages, microbatches, base)
    cap = _live(stages, microbatches, 0) * base
    for s, b in enumerate(bits):
        live = _live(stages, microbatches, s)
        ok = [w for w in WIDTHS if w >= base and live * w <= cap]
        assert b == max(ok)
        assert live * b <= cap                          # no stage exceeds the fullest one


def test_closed_cases():
    assert agoq.agoq_dbca_pp_bits(4, 8) == [4, 5, 8, 8]      # live 4,3,2,1; cap 16
    assert agoq.agoq_dbca_pp_bits(8, 8) == [4, 4, 5, 6, 8, 8, 8, 8]
    assert agoq.agoq_dbca_pp_bits(4, 2) == [4, 4, 4, 8]      # fewer micro-batches than stages
    assert agoq.agoq_dbca_pp_bits(1, 1) == [4]
    assert agoq.agoq_dbca_pp_bits(3, 4, base_bits=8) == [8, 8, 8]


def test_widths_never_decrease_along_the_pipeline():
    for stages, mb in itertools.product(range(1, 12), (1, 3, 7, 64)):
        bits = agoq.agoq_dbca_pp_bits(stages, mb)
        assert all(a <= b for a, b in zip(bits, bits[1:]))


def test_rejects_bad_arguments():
    with pytest.raises(agoq.AgoqError):
        agoq.agoq_dbca_pp_bits(0, 4)
    with pytest.raises(agoq.AgoqError):
        agoq.agoq_dbca_pp_bits(4, 0)
    with pytest.raises(agoq.AgoqError):
        agoq.agoq_dbca_pp_bits(4, 4, base_bits=7)
