"""The fused-path trace summary (run_op --trace) on fabricated records: task
spans, per-tile time and per-window block occupancy (host logic only)."""
import torch

from dispatch_ffn_combine_gb300.run_op import trace_summary


def _rec(block, kind, tiles, start_ns, end_ns):
    return [block, kind, 0, tiles, start_ns & 0xFFFFFFFF, start_ns >> 32, end_ns & 0xFFFFFFFF, end_ns >> 32]


def test_trace_summary_spans_tiles_and_windows():
    base = 5 << 32  # timestamps above 2^32 ns exercise the high word
    recs = [
        _rec(0, 3, 0, base + 0, base + 10_000),          # dispatch 0-10 us
        _rec(1, 6, 4, base + 10_000, base + 50_000),      # gemm session, 4 tiles in 40 us
        _rec(0, 6, 6, base + 10_000, base + 70_000),      # gemm session, 6 tiles in 60 us
        _rec(1, 5, 0, base + 70_000, base + 100_000),     # combine 70-100 us
    ]
    tr = torch.tensor(recs, dtype=torch.int64).to(torch.int32)
    lines = trace_summary(tr, len(recs), windows=10)
    assert lines[0] == "records 4, span 100.0 us"
    gemm = next(s for s in lines if s.strip().startswith("gemm"))
    assert "tiles 10, 10.0 us per tile" in gemm
    assert "first start      10.0 us" in gemm and "last end      70.0 us" in gemm
    disp = next(s for s in lines if s.strip().startswith("dispatch"))
    assert "mean      10.0 us" in disp
    rows = [s.split() for s in lines if s.strip() and s.strip()[0].isdigit()]
    assert len(rows) == 10
    occ = [[float(v) for v in r[1:]] for r in rows]  # columns: dispatch, combine, gemm (kinds sorted 3, 5, 6)
    assert occ[0] == [1.0, 0.0, 0.0]
    assert occ[3] == [0.0, 0.0, 2.0]
    assert occ[6] == [0.0, 0.0, 1.0]
    assert occ[9] == [0.0, 1.0, 0.0]


def test_trace_summary_caps_at_buffer_and_handles_empty():
    assert trace_summary(torch.zeros((0, 8), dtype=torch.int32), 0) == ["no task records"]
    tr = torch.tensor([_rec(0, 2, 0, 0, 1000)], dtype=torch.int32)
    assert trace_summary(tr, 5)[0].startswith("records 1,")  # more tasks ran than the buffer held
