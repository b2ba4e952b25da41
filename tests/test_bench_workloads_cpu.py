"""The default benchmark line's 'workloads' block contains its failures: an entry
that cannot run records its error and the block (and so the main line) is still
returned. Run on the CPU, where every device call fails, with the tiny head in
place of the large ones so that the host draws take no time."""
import pytest

import bench

torch = pytest.importorskip("torch")


def test_failing_entries_record_their_error(monkeypatch):
    import flce_inputs
    import linear_cross_entropy_flce_gb300 as flce

    monkeypatch.setattr(bench, "OTHER_WORKLOADS", ("tiny",))
    wl = flce_inputs.get("tiny")
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    dev = torch.device("cpu")
    H = torch.from_numpy(Hb.view("int16")).view(torch.bfloat16)
    W = torch.from_numpy(Wb.view("int16")).view(torch.bfloat16)
    lab = torch.from_numpy(y)

    class Args:
        other_steps = 2

    block = bench.other_workloads(Args(), flce, H, W, lab, wl, dev, 0, None,
                                  {"bf16_tflops": 1910.7})
    assert "note" in block
    for key in ("tiny", "tiny_forward_only", "tiny_fp8"):
        assert set(block[key]) == {"error"}, block[key]
        assert block[key]["error"]

