"""The pipe-peak probes (os2_peak_probe) compute what they claim: the
tcgen05 kind::f16 probes (1-SM and 2-SM) and the mma.sync s8 probe give the
exact product of their formula operands on every entry, so their timed runs
measure real tensor-core work."""
import pytest

import rns_emulated_fp64_gb300 as os2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", [os2.PROBE_F16_1SM, os2.PROBE_F16_2SM, os2.PROBE_S8_SYNC])
@pytest.mark.parametrize("iters", [1, 37])
def test_peak_probe_results_exact(kind, iters):
    flop, bad, ctas = os2.peak_probe(kind, iters, check=True)
    assert os2.get_status() == 0
    assert ctas > 0
    assert bad == 0, f"{bad} mismatching entries"
    assert flop > 0
    assert os2.peak_probe(kind, 2 * iters) == pytest.approx(2 * flop)
    assert os2.get_status() == 0
