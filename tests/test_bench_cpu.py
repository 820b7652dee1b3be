"""The benchmark's CPU oracle legs on tiny seeded cases (no GPU): the decode and
prefill baselines run the fp64 oracle and report a positive rate in the units of
their GPU lines, with the sample they timed."""
import bench
import msa_inputs as mi


def test_cpu_baseline_decode_reports_requests_per_second():
    _, dec = mi.tiny_case(seed=1000, device="cpu")
    out = bench.cpu_baseline_decode(0, budget_s=0.2, max_reqs=8, case=dec)
    assert out["unit"] == "tok/s" and out["kind"] == "oracle" and out["cores"] == 1
    assert out["value"] > 0 and "decode requests" in out["sample"]


def test_cpu_baseline_prefill_reports_rows_per_second():
    pre, _ = mi.tiny_case(seed=1000, device="cpu")
    out = bench.cpu_baseline_prefill(pre, budget_s=0.2, max_rows=16)
    assert out["unit"] == "q-tok/s" and out["kind"] == "oracle" and out["cores"] == 1
    assert out["value"] > 0 and "rows spread over" in out["sample"]
