"""The benchmark's algorithmic byte and FLOP counts per unit of work, written
out from the entry sizes (288 B per FP4 main entry, 72 B per FP4 indexer
entry, 68 B for the write-ups' indexer entry, 1024 B per bf16 window row,
528 B per MXFP8 one) and the per-query attention traffic, and the workload
list the benchmark and the tests share."""
import bench
import synth


def test_attention_bytes_per_query_token():
    # 512 top-k entries x 288 B + 128 window rows x 1024 B + 64 x 512 bf16 Q
    # + 64 x 512 fp32 out + 512 int32 ids
    assert bench.attend_query_bytes("fp4") == 512 * 288 + 128 * 1024 + 65536 + 131072 + 2048 == 477184
    assert bench.attend_query_bytes("fp4", row_bytes=528) == 512 * 288 + 128 * 528 + 65536 + 131072 + 2048
    assert bench.attend_query_bytes("bf16", 512, 128) == 512 * 1024 + 128 * 1024 + 65536 + 131072 + 2048


def test_indexer_entry_and_window_row_bytes():
    wl = synth.WORKLOADS["decode_b8_ctx32768_r2_fp4"]
    assert bench.idx_entry_bytes(wl) == 72 and bench.swa_row_bytes(wl) == 1024
    wf = synth.WORKLOADS["decode_b8_ctx32768_r2_fp4_idx68_fp8swa"]
    assert bench.idx_entry_bytes(wf) == 68 and bench.swa_row_bytes(wf) == 528


def test_index_chunk_takes_every_query_within_the_budget():
    assert bench.index_chunk(2 << 20, 4096) == 4096             # 8 GiB of workspace: one pass
    assert bench.index_chunk(2 << 20, 4096, budget=1 << 30) == 512
    assert bench.index_chunk(1 << 40, 7) == 1                    # at least one query per pass


def test_workloads_are_consistent():
    for name, wl in synth.WORKLOADS.items():
        assert wl.name == name
        assert wl.ctx % wl.ratio == 0
        if wl.tq > 1:
            assert wl.entries == (wl.ctx + wl.tq) // wl.ratio
        else:
            assert wl.entries == wl.ctx // wl.ratio
        assert not (wl.idx68 and wl.cache != "fp4")
    assert bench.DEFAULT_WORKLOAD in synth.WORKLOADS


def test_traffic_figures_match_their_profile_summaries():
    # every DRAM traffic figure the benchmark reports is the sum of the
    # dram__bytes_read + dram__bytes_write rows of the summaries it names
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for wl, stages in bench.TRAFFIC.items():
        assert wl in synth.WORKLOADS
        for stage, (traffic, sources) in stages.items():
            total = 0
            for src in sources.split(" + "):
                text = open(os.path.join(root, src)).read()
                m = re.search(r"dram__bytes_read\.sum \+ dram__bytes_write\.sum \| ([\d,]+) B \+ ([\d,]+) B", text)
                assert m, src
                total += int(m.group(1).replace(",", "")) + int(m.group(2).replace(",", ""))
            assert total == traffic, (wl, stage, total, traffic)
