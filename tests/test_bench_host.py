"""Host-side arithmetic of bench.py, without a GPU: the decode roofline's byte
counts against the pages' model size, the peak the roofline divides by, and
the command-line defaults the timing rules need."""
import json

import pytest

import bench
from q8_quantized_llama_gb300 import synth


def _extras(cfg):
    """Bytes decode_bytes adds beyond the Q8_0 projections and lm_head: the
    f32 norm weights of every layer and the final norm, and the embedding row
    of the step's token."""
    h = cfg["n_embd"]
    return cfg["n_layer"] * 8 * h + 4 * h + bench.q8_bytes(1, h)


def test_decode_bytes_135m_match_the_pages_model_size():
    """The projections and the tied lm_head of the 135M model are the 136.3 MiB
    of Q8_0 weights the pages give for the file's weights ("速度", CPU GGUF);
    K and V rows cost 46,080 bytes per cached position (30 layers x 3 heads x
    64 dims x 4 bytes x 2)."""
    cfg = synth.MODEL_135M
    w, kv = bench.decode_bytes(cfg, 1.0)
    proj = w - _extras(cfg)
    assert proj == 142_884_864
    assert round(proj / 2**20, 1) == 136.3
    assert kv == 46_080


def test_decode_bytes_7b():
    cfg = synth.MODEL_7B
    w, kv = bench.decode_bytes(cfg, 1.0)
    assert w - _extras(cfg) == 7_554_793_472            # 32 layers + untied head, 34 bytes per 32 weights
    assert kv == 262_144                                # 32 x 8 heads x 128 dims x 4 bytes x 2


def test_hbm_peak_reads_the_measured_file(tmp_path, monkeypatch):
    # a measured-peaks file with a known copy bandwidth: the measured branch
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6543.2, "bf16_tflops": 1900.0}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peak, kind = bench.hbm_peak()
    assert kind == "measured" and peak == pytest.approx(6543.2)
    # no file: the stated fallback
    empty = tmp_path / "empty"
    empty.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(empty))
    peak, kind = bench.hbm_peak()
    assert kind == "fallback" and peak == bench.FALLBACK_HBM_GBS


def test_defaults_follow_the_timing_rules():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1 and a.impl == "ours"
    assert bench.aggregate_throughput(100.0, 2.0, 1) == (50.0, 2.0)
