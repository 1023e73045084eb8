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
