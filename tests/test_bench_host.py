"""Host-side pieces of bench.py that shape the reported numbers: the
roofline peaks per format, the quantization step's byte count, the
whole-job throughput of replicas and the profile traffic lookup."""
import pytest

import bench
from precision_attention_diffusion_sage_gb300.inputs import WORKLOADS


def test_roofline_peaks_per_format():
    p16 = 1911.5  # measured dense BF16 (FP16 runs at the same rate)
    # INT8 codes on the FP16 pipe for Q K^T, FP8 P V at twice the rate: harmonic mean
    assert bench._roofline_peak(p16, 0) == pytest.approx(2 / (1 / p16 + 1 / (2 * p16)))
    assert bench._roofline_peak(p16, 0) == pytest.approx(2548.67, abs=0.01)
    assert bench._roofline_peak(p16, 2) == pytest.approx(3823.0)           # both halves FP8
    assert bench._roofline_peak(p16, 1) == pytest.approx(5734.5)           # FP4 QK, FP8 PV
    assert bench._roofline_peak(p16, 3) == bench._roofline_peak(p16, 1)    # rotated MXFP4
    assert bench._roofline_peak(p16, 4) == pytest.approx(11469.0)          # both halves FP4


def test_clock_peak_from_measured_mma_rates():
    """The informational peak at the sampled clock: measured FLOP/clk/SM of
    each MMA kind (f16 8192, f8 16384, f4 32768) x 152 SMs x MHz, halves
    combined harmonically; INT8 at 2070 MHz is 10922.7 x 152 x 2.07e9."""
    assert bench._clock_peak(0, 2070) == pytest.approx(2 / (1 / 8192 + 1 / 16384) * 152 * 2.07e-3)
    assert bench._clock_peak(0, 2070) == pytest.approx(3436.71, abs=0.01)
    assert bench._clock_peak(2, 2070) == pytest.approx(16384 * 152 * 2.07e-3)
    assert bench._clock_peak(4, 1000) == pytest.approx(32768 * 152 * 1e-3)
    assert bench._clock_peak(0, 1035) == pytest.approx(bench._clock_peak(0, 2070) / 2)


def test_quant_bytes_by_element_count():
    """Bytes per input element, from what each pass reads and writes: INT8
    Q and K read 2 and write 2 (FP16-held codes), V read twice (maxima, then
    encoding) and written once as FP8; MXFP4 V is one pass of 2 bytes in and
    0.5 + 1/32 out, like MXFP4 Q and K."""
    w = WORKLOADS["image_dit"]  # N = 4608 = 36 x 128: no padding
    elems = w.B * w.H * w.Nq * w.D
    assert bench._quant_bytes(w, w.Nq, w.Nk) == pytest.approx(13 * elems)
    w4 = WORKLOADS["mxfp4_v4_self"]
    e4 = w4.B * w4.H * w4.Nq * w4.D
    assert bench._quant_bytes(w4, w4.Nq, w4.Nk) == pytest.approx(3 * (2 + 0.5 + 1 / 32) * e4)


def test_replica_throughput_is_whole_job():
    # two replicas, 1e12 FLOP each per step, 10 steps, the slower took 1 s in total
    assert bench.replica_throughput(1e12, 10, 1000.0, 2) == pytest.approx(20.0)
    assert bench.replica_throughput(1e12, 10, 1000.0, 1) == pytest.approx(10.0)


def test_profiled_traffic_needs_the_current_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k.md").write_text(
        "text\n`traffic: kernel=sage_attn_kernel<0,2,2> workload=image_dit "
        "sources_sha256=abc dram_bytes_per_launch=123`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "_kernel_sources_sha256", lambda: "abc")
    assert bench._profiled_traffic("sage_attn_kernel<0,2,2>", "image_dit") == 123
    assert bench._profiled_traffic("sage_attn_kernel<0,2,2>", "video_dit") is None
    monkeypatch.setattr(bench, "_kernel_sources_sha256", lambda: "changed")
    assert bench._profiled_traffic("sage_attn_kernel<0,2,2>", "image_dit") is None

