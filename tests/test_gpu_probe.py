"""The FMA-throughput probe that gives the arithmetic rooflines their
denominators (include/swe_probe.h): each kind returns a rate within a factor
of a few of the GB300 data sheet (152 SMs x 128 FP32 lanes x 2 flops at up to
2.07 GHz = 80.5 TFLOP/s; FP64 about 1.25 TFLOP/s), the timed launch lasts
about as long as asked, and packed FP32 pairs are no slower than scalar FMAs."""
import pytest

from finite_volume_shallow_gb300 import swe as S

pytestmark = pytest.mark.gpu


def test_fma_probe_rates_are_plausible():
    rates = {}
    for kind in (S.PROBE_FFMA, S.PROBE_FFMA2, S.PROBE_DFMA):
        rate, ms = S.swe_probe_fma_rate(kind, 30.0)
        assert 10.0 <= ms <= 120.0, (kind, ms)
        rates[kind] = rate / 1e12
    assert 20.0 <= rates[S.PROBE_FFMA] <= 120.0, rates
    assert 20.0 <= rates[S.PROBE_FFMA2] <= 240.0, rates
    assert rates[S.PROBE_FFMA2] >= 0.8 * rates[S.PROBE_FFMA], rates
    assert 0.2 <= rates[S.PROBE_DFMA] <= 10.0, rates


def test_fma_probe_rejects_bad_arguments():
    for kind, ms in ((7, 10.0), (S.PROBE_DFMA, 0.0), (S.PROBE_FFMA, 5000.0)):
        with pytest.raises(S.SweError) as e:
            S.swe_probe_fma_rate(kind, ms)
        assert e.value.status == S.SWE_ERR_ARG
