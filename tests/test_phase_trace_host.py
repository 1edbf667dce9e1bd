"""Host logic of the phase-trace diagnostic (CPU only): call parsing, byte counts and the report
tables, on a synthetic trace whose phase times are known."""
import importlib

import numpy as np
import pytest
import torch

pt = importlib.import_module("nvfp4_weight_only_gemv_gb300.phase_trace")


def test_parse_call():
    assert pt.parse_call("dense:4096:1024:5:bf16") == {"kind": "dense", "N": 4096, "K": 1024, "M": 5, "bf16": True}
    c = pt.parse_call("moe:288:3072:4096:4:8:0")
    assert (c["E"], c["N"], c["K"], c["T"], c["top_k"], c["xps"]) == (288, 3072, 4096, 4, 8, False)
    with pytest.raises(SystemExit):
        pt.parse_call("conv:1:2:3")


def test_algorithmic_bytes_match_the_stated_formula():
    # N*K*(0.5 + 1/16) + M*K*2 + M*N*out_bytes: the attention projection and the FFN gate/up pair
    assert pt.alg_bytes(pt.parse_call("dense:4096:4096:1:bf16"), None) == 9_453_568
    assert pt.alg_bytes(pt.parse_call("gate_up:12288:4096:1"), None) == 56_729_600


def synthetic_trace():
    """Two launches of four CTAs: entry 1 us, dependency 3 us, x staged 4 us, first box 4.5 us,
    stores at 9, 9, 9 and 12 us, exit 0.1 us after the store; SM clock 2 GHz."""
    tr = np.zeros((16, 1024, 40), dtype=np.int64)
    for launch, shift in ((0, 0), (1, 20_000)):
        for cta, stored in enumerate((9_000, 9_000, 9_000, 12_000)):
            row = tr[launch, cta]
            times = {0: 1_000, 1: 1_500, 2: 3_000, 3: 4_000, 4: 4_500, 5: stored - 200, 6: stored, 7: stored + 100}
            for ph, t in times.items():
                row[2 * ph] = t + shift
                row[2 * ph + 1] = 2 * (t - 1_000)  # clock64 at 2 GHz from entry
            row[24] = 10 + cta                  # the SM
            row[38] = row[7] + 800              # dense: just before the first box wait
            row[39] = row[38] + 200             # just after it
    return torch.from_numpy(tr)


def test_report_tables_on_a_synthetic_trace():
    meta = [("dense:4096:4096:1:bf16", 9_453_568), ("dense:4096:4096:1:bf16", 9_453_568)]
    lines = pt.summarise(synthetic_trace(), 2, meta)
    text = "\n".join(lines)
    # per-CTA phase durations: entry->dep 2, dep->x 1, x->box 0.5, box->stored (median) 4.5,
    # stored->exit 0.1 us, at 2 GHz
    rows = [l.split()[1:] for l in lines if l.startswith("dense") and len(l.split()) == 7]
    assert rows[0] == ["2.00", "1.00", "0.50", "4.50", "0.10", "2.00"] and rows[1] == rows[0]
    # the store tail: the 90th percentile of (9, 9, 9, 12) is 11.1 us, the last 12 us, and the
    # last CTA ran on SM 13
    tail = [l for l in lines if l.startswith("dense") and l.split()[-1] == "13"]
    assert len(tail) == 2 and tail[0].split()[1:3] == ["2.10", "3.00"]
    # the dense clock table: 800 cycles of set-up, a 200-cycle wait, no landing mark (word 36)
    dense = [l for l in lines if l.startswith("dense") and l.split()[1:3] == ["800", "200"]]
    assert len(dense) == 2 and dense[0].split()[3:] == ["-", "-"]
    assert "x_staged->box wait" in text and "stored p90-med" in text


def test_landing_mark_column():
    tr = synthetic_trace().numpy().copy()
    tr[0, :4, 36] = tr[0, :4, 4] - 50  # first box landed 50 ns before the dependency release
    lines = pt.summarise(torch.from_numpy(tr), 2, [("dense:1:2:3", 1), ("dense:1:2:3", 1)])
    dense = [l for l in lines if l.startswith("dense") and l.split()[1:3] == ["800", "200"]]
    # issued (phase 1) -> landed: 3000 - 50 - 1500 ns; landed -> dependency release: 50 ns
    assert dense[0].split()[3:] == ["1.45", "0.05"]
    assert dense[1].split()[3:] == ["-", "-"]
