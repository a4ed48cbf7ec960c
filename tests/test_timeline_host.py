"""The timeline profiling aid's summary, on synthetic per-CTA rows (CPU only; the
timeline build itself runs on the GPU)."""
import numpy as np

from paged_kv_cache_252_gb300 import timeline, workloads as wl


def test_summary_of_synthetic_rows():
    base = 10_000_000
    rows = np.zeros((4, timeline.NEV), np.uint64)
    for i in range(4):
        # entry, planned, first/last issue, first/last data, exit (ns)
        ev = [0, 500, 900, 9000 + 100 * i, 2000, 9500 + 100 * i, 10000 + 1000 * i]
        rows[i, :7] = [base + e for e in ev]
        rows[i, 7] = (i + 3) | (2 << 16) | (40 << 32)
        rows[i, 8] = base + ev[5] + 300          # last piece's output written
        rows[i, 9] = base + ev[5] + 800          # counted
    s = timeline.summarize(wl.tiny(), rows)
    assert "4 CTAs (4 with work)" in s
    assert "span (first entry to last exit): 13.00 us" in s
    assert "ramp (median first data): 2.00 us" in s
    assert "blocks per CTA: min 40, median 40, max 40" in s
    assert "pieces per CTA: min 2, median 2, max 2" in s
    assert "| piece_out - last_data (4 CTAs) | 0.30 | 0.30 | 0.30 | 0.30 | 0.30 |" in s
    assert "| counted - last_data (4 CTAs) | 0.80 |" in s
