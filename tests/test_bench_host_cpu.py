"""bench.py's host arithmetic against closed forms of the workloads: the
algorithmic bytes and flops that the roofline divides by, and the roofline
fraction itself.  No GPU; the cases carry only the fields that arithmetic
reads (the full generators would allocate gigabytes)."""
import types

import numpy as np
import pytest

import bench
import workloads as W

PEAKS = {"hbm_gbs": 6786.6, "bf16_tflops": 1877.6, "source": "measured"}


def _case(name, kind, seq_lens, K=2048):
    """Latent 64x576/512 shapes with the 64x128 FP8 indexer."""
    seq_lens = np.asarray(seq_lens, np.int32)
    if kind == "prefill":
        q_pos = np.arange(int(seq_lens[0]), dtype=np.int32)
    else:
        q_pos = (seq_lens - 1).astype(np.int32)
    return types.SimpleNamespace(name=name, kind=kind, seq_lens=seq_lens,
                                 n_elig=(q_pos + 1).astype(np.int32), K=K, Hq=64, Dqk=576,
                                 Dv=512, latent=True, Dkv=576, H_i=64, D_i=128, idx_dtype="fp8")


def test_prefill_flops_are_the_causal_and_selected_pair_counts():
    T, K = 16384, 2048
    a = bench.algorithmic(_case("prefill", "prefill", [T], K))
    pairs = T * (T + 1) // 2                       # every p <= t
    selected = K * (K + 1) // 2 + (T - K) * K      # sum over t of min(t + 1, K)
    assert (pairs, selected) == (134_225_920, 31_458_304)
    assert a["index_flops"] == 2.0 * pairs * 64 * 128
    assert a["attn_flops"] == 2.0 * selected * 64 * (576 + 512)
    assert a["index_flops"] == pytest.approx(2.199e12, rel=1e-3)
    assert a["attn_flops"] == pytest.approx(4.381e12, rel=1e-3)


def test_decode_bytes_are_keys_plus_selected_rows():
    # million: 2^20 positions of 128-byte FP8 keys per sequence, 2048 latent rows
    a = bench.algorithmic(_case("million", "decode", [1 << 20] * 8))
    assert a["index_bytes"] == 8 * (1 << 20) * 128 == 1_073_741_824
    assert a["gather_bytes"] == 8 * 2048 * 1152 == 18_874_368
    # long-dec: 655,360 positions in all
    a = bench.algorithmic(_case("long-dec", "decode", [262144, 196608, 131072, 65536]))
    assert a["index_bytes"] + a["gather_bytes"] == 655_360 * 128 + 4 * 2048 * 1152 == 93_323_264
    # dec-batch: the generator's lengths, every one above K
    L = W.dec_batch_lens()
    assert L.shape == (32,) and L.min() >= 8192 and L.max() <= 32768
    a = bench.algorithmic(_case("dec-batch", "decode", L))
    assert a["index_bytes"] == int(L.astype(np.int64).sum()) * 128
    assert a["gather_bytes"] == 32 * 2048 * 1152 == 75_497_472
    # a context shorter than K gathers only its own rows
    a = bench.algorithmic(_case("short", "decode", [100, 5000]))
    assert a["gather_bytes"] == (100 + 2048) * 1152


def test_roofline_takes_the_slower_stage_and_its_peak():
    # decode: attention is the slower stage; gathered bytes over its time
    c = _case("dec-batch", "decode", W.dec_batch_lens())
    roof, step_bytes = bench.roofline_of({"case": c, "stage_ms": [0.0233, 0.0210, 0.0533]}, PEAKS)
    want = 75_497_472 / 0.0533e-3 / 1e9
    assert (roof["kernel"], roof["bound"], roof["unit"]) == ("sparse_attn", "hbm", "GB/s")
    assert roof["achieved"] == pytest.approx(want, abs=0.1)
    assert roof["frac"] == pytest.approx(want / 6786.6, abs=1e-4)
    assert step_bytes == bench.algorithmic(c)["index_bytes"] + 75_497_472
    # prefill: tensor-bound; attention against the bf16 peak...
    p = _case("prefill", "prefill", [16384])
    roof, _ = bench.roofline_of({"case": p, "stage_ms": [1.39, 0.58, 12.78]}, PEAKS)
    assert (roof["kernel"], roof["bound"]) == ("sparse_attn", "tensor")
    assert roof["achieved"] == pytest.approx(4.381e12 / 12.78e-3 / 1e12, rel=1e-3)
    assert roof["peak"] == pytest.approx(1877.6)
    # ...and an FP8 indexer, when it is the slower stage, against twice that
    roof, _ = bench.roofline_of({"case": p, "stage_ms": [20.0, 0.58, 12.78]}, PEAKS)
    assert roof["kernel"] == "index_score"
    assert roof["peak"] == pytest.approx(2 * 1877.6)
    assert roof["frac"] == pytest.approx(2.199e12 / 20e-3 / 1e12 / (2 * 1877.6), rel=1e-3)


def test_headline_line_carries_the_contract_keys():
    """The JSON line built from a (fake) measurement: every key the bench
    contract names, whole-job throughput, and the roofline objects."""
    c = _case("dec-batch", "decode", W.dec_batch_lens())
    c.B, c.Nq, c.bs = 32, 32, 64
    steps, total_ms = 20, 20 * 0.0861
    res = {"case": c, "total_ms": total_ms, "stage_ms": [0.0233, 0.0210, 0.0533],
           "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []},
           "e2e": {k: {"value": 2.6e5, "unit": "queries/s", "h2d_bytes_per_step": 2694656,
                       "d2h_bytes_per_step": 2097152} for k in ("calls", "graph")},
           "launches": 80, "launches_per": {"step": 4}, "status": 0, "cache_write": None}
    args = types.SimpleNamespace(steps=steps, warmup=5)
    for world in (1, 2):
        line = bench.headline(args, world, res, PEAKS)
        for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                  "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                  "roofline", "clocks", "e2e", "gpu_launches"):
            assert k in line, k
        assert line["metric"] == "decode queries/sec" and line["unit"] == "queries/s"
        assert line["higher_is_better"] is True and line["scaling"] == "weak"
        assert line["vs_baseline"] is None and line["n_gpus"] == world
        # whole job: every rank's 32 queries over the slowest rank's time
        assert line["value"] == pytest.approx(32 * world * steps / (total_ms / 1e3))
        assert line["ms_per_step"] == pytest.approx(0.0861)
        assert line["config"]["workload"] == "dec-batch"
        assert line["config"]["parallelism"] == ("1gpu" if world == 1 else "replicas2")
        assert "flushed" in line["config"]["l2"]
        for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
            assert k in line["roofline"], k
        for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
            assert k in line["e2e"], k
        assert line["path_roofline"]["algorithmic_bytes_per_step"] == \
            bench.algorithmic(c)["index_bytes"] + 75_497_472
