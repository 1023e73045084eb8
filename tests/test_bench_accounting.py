"""The benchmark's byte accounting on CPU: the algorithmic bytes per launch
follow the per-element formulas of the path (bf16 in, one code byte and two
fp32 scalars per block out, P compressed shards in for the reduce, fp32 out
of the decompress), and the committed DRAM-traffic record is reported only
while the codec sources still match the digest it was taken on."""

import json

import pytest

import bench

HEADLINE_ELEMS = 8192 * 4096  # one shard of the GPT-6.7B-shaped workload


@pytest.mark.parametrize("P,block", [(4, 128), (8, 256), (2, 128), (16, 256)])
def test_algorithmic_bytes_per_element(P, block):
    n = 1024 * block
    b = bench.algorithmic_bytes(P, n, block)
    assert b["compress"] == P * n * (2 + 1 + 8 / block)
    assert b["reduce"] == n * (P + 1) * (1 + 8 / block)
    assert b["decompress"] == n * (1 + 8 / block + 4)
    f = bench.algorithmic_bytes(P, n, block, fused=True)
    assert f["compress"] == b["compress"]
    # the one-call minimum does not re-read the compressed sum
    assert f["reduce_decompress"] == b["reduce"] + b["decompress"] - n * (1 + 8 / block)
    assert bench.algorithmic_bytes(P, n, block, out_bytes=2)["decompress"] == n * (1 + 8 / block + 2)


def test_headline_step_bytes():
    b = bench.algorithmic_bytes(4, HEADLINE_ELEMS, 128)
    assert b == {"compress": 411_041_792, "reduce": 178_257_920, "decompress": 169_869_312}
    assert sum(b.values()) == 759_169_024


def test_traffic_record_is_dropped_when_the_sources_change(tmp_path, monkeypatch):
    rec = {"dram_bytes_per_launch": 123, "source_digest": bench.kernel_source_digest()}
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.committed_traffic() == 123
    rec["source_digest"] = "0" * 16
    f.write_text(json.dumps(rec))
    assert bench.committed_traffic() is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.committed_traffic() is None


def test_codec_bytes_of_the_round_trip_leg():
    n = 4096 * 2560  # the GPT-2.7B-shaped activation
    b = bench.codec_bytes(n, 128)
    assert b["compress"] == n * (2 + 1 + 8 / 128)
    assert b["decompress"] == n * (1 + 8 / 128 + 4)
    assert bench.codec_bytes(n, 256, out_bytes=2)["decompress"] == n * (1 + 8 / 256 + 2)


def test_kernel_sample_summary_reports_count_and_spread():
    st = bench.summarize([0.070, 0.069, 0.071, 0.090])
    assert st["samples"] == 4
    assert st["us_min"] == pytest.approx(69.0) and st["us_max"] == pytest.approx(90.0)
    assert st["us_mean"] == pytest.approx(75.0) and st["us_median"] == pytest.approx(70.5)
    e = bench.kernel_entry(0.075, 411_041_792, 6780.0, **st)
    assert e["gbs"] == pytest.approx(411_041_792 / 75e-6 / 1e9)
    assert e["frac_of_peak"] == pytest.approx(e["gbs"] / 6780.0) and e["samples"] == 4


def test_spec_peak_is_always_reported():
    gbs, src = bench.spec_hbm_gbs(0)
    assert gbs > 0 and src
    # without a GPU (this host) the nominal GB300 figure stands in
    import torch

    if not torch.cuda.is_available():
        assert gbs == bench.SPEC_NOMINAL_GBS and "nominal" in src


@pytest.mark.parametrize("world", [2, 4, 8])
def test_exchange_bytes_split_the_local_path_across_ranks(world):
    # W ranks of one [8192, 4096] activation each: together they compress
    # what the one-GPU path compresses for P = W shards, each reduces 1/W of
    # the rows over W shards, and each decompresses the whole sum
    rows, d, block = 8192, 4096, 128
    e = bench.exchange_bytes(world, rows, d, block)
    local = bench.algorithmic_bytes(world, rows * d, block)
    assert world * e["compress"] == local["compress"]
    assert world * e["reduce"] == local["reduce"]
    assert e["decompress"] == local["decompress"]
    # a ragged split pads the last chunk: the padded rows are reduced and
    # decompressed too
    r = bench.exchange_bytes(3, 100, 256, 128)
    assert r["reduce"] == 4 * (34 * 256 + 8 * 34 * 2)
    assert r["decompress"] == 3 * (34 * 256 * 5 + 8 * 34 * 2)
    # pieces of a chunk: its rows are rounded up to a multiple of the stages
    assert bench.exchange_bytes(3, 100, 256, 128, stages=4)["reduce"] == 4 * (36 * 256 + 8 * 36 * 2)
    assert bench.exchange_bytes(4, 8192, 4096, 128, stages=4) == bench.exchange_bytes(4, 8192, 4096, 128)
