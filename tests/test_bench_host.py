"""Host logic of bench.py without a GPU: the N-rank aggregation over gloo (world size 2), seeds,
byte models, the clock-log parser, the staleness rule for profiled traffic, the CPU model and the
accuracy record."""
import json
import os
import socket

import numpy as np
import pytest

import bench
import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, n, lr = bench.dist_env()
    # each rank: its own batch (own seed), its own bytes and time; the job sums bytes, maxes time
    w = W.make_config(2, seed=bench.rank_seed(2, r), B=3, ctx_lo=20, ctx_hi=80)
    local_bytes = W.kv_bytes(w) * 10
    local_ms = 5.0 + 3.0 * r
    tot, mx = bench.aggregate(local_bytes, local_ms)
    q.put((r, n, lr, local_bytes, tot, mx, int(w.q.view(np.uint16)[0, 0, 0])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, n0, l0, b0, t0, m0, q0), (r1, n1, l1, b1, t1, m1, q1) = res
    assert (r0, r1, n0, n1, l0, l1) == (0, 1, 2, 2, 0, 1)
    assert t0 == t1 == b0 + b1
    assert m0 == m1 == 8.0
    assert q0 != q1  # the ranks decode different batches (weak scaling)


def test_single_process_aggregate_is_identity():
    assert bench.aggregate(123.0, 4.5) == (123.0, 4.5)


def test_attention_bytes_exclude_the_write():
    w = W.make_config(2, B=4, ctx_lo=100, ctx_hi=200)
    wr = 4 * w.Hkv * w.D * 2 * 2 * 2 + 8 * 4  # K+V rows read and written per token, slot ids
    assert bench.attention_bytes(w) == W.kv_bytes(w) - wr
    tokens = int(w.context_lens.sum())
    assert bench.attention_bytes(w) >= tokens * w.Hkv * w.D * 2 * 2


def test_prefix_bytes_count_the_shared_prefix_once():
    w = W.make_config(5, B=4, ctx_lo=16, ctx_hi=40, prefix_tokens=64)
    logical = W.kv_bytes(w, unique=False)
    unique = W.kv_bytes(w)
    assert logical - unique == 3 * 64 * w.Hkv * w.D * 2 * 2


def test_clock_rows_parser():
    rows = ["0, 1965, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
            "0, 1980, 2070, 950.3, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
            "0, 1950, 2070, 951.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"]
    c = bench.parse_clock_rows(rows)
    assert c == {"sm_mhz": 1965.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert bench.parse_clock_rows(["garbage"]) is None


def test_profiled_traffic_is_null_when_sources_changed(tmp_path, monkeypatch):
    import json
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench.profiled_traffic("x") is None                     # no data file
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({"split_kernel": {"x": {"kernel_source_sha": "deadbeef",
                                                    "traffic_bytes_per_launch": 1234}}}))
    assert bench.profiled_traffic("x") is None                     # captured on other sources
    f.write_text(json.dumps({"split_kernel": {"x": {"kernel_source_sha": bench.kernel_source_hash(),
                                                    "traffic_bytes_per_launch": 1234}}}))
    assert bench.profiled_traffic("x") == 1234
    assert bench.profiled_traffic("y") is None                     # no capture of that workload


def test_committed_traffic_file_covers_the_bench_workloads():
    import json
    import os
    with open(os.path.join(bench.PROFILES, "traffic.json")) as fh:
        d = json.load(fh)["split_kernel"]
    for name in ("llama3_8b_gqa", "long_splitk", "int8_kv", "prefix_shared"):
        assert int(d[name]["traffic_bytes_per_launch"]) > 0
        assert len(d[name]["kernel_source_sha"]) == 16


def test_source_fingerprint_ignores_comments_and_layout_only():
    code = 'int f(int x) {\n    return x + 1;  // one more\n}\nconst char* s = "a // b";\n'
    relaid = '/* header */\nint f(int x) { return x + 1; }\n\nconst char* s = "a // b";'
    assert bench.source_code_only(code) == bench.source_code_only(relaid)
    # code, and text inside literals, still count
    assert bench.source_code_only(code) != bench.source_code_only(code.replace("x + 1", "x + 2"))
    assert bench.source_code_only(code) != bench.source_code_only(code.replace('"a // b"', '"a // c"'))


def test_launch_count_model():
    w = W.make_config(2, B=2, ctx_lo=100, ctx_hi=200)
    assert bench.cuda_launches_per_step(w, 512) == 2      # one split: no merge launch
    assert bench.cuda_launches_per_step(w, 16) == 3


@pytest.mark.parametrize("cfg", [2, 4])
def test_reference_leg_runs(cfg, capsys):
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0", "--config", str(cfg)])
    import json
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_cpu_model_parser():
    x86 = "processor\t: 0\nvendor_id\t: GenuineIntel\nmodel name\t: Intel(R) Xeon(R) Platinum 8480+\n"
    assert bench.parse_cpu_model(x86, "x86_64") == "Intel(R) Xeon(R) Platinum 8480+"
    grace = "processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n"
    assert bench.parse_cpu_model(grace, "aarch64") == "Arm Neoverse-V2"
    other = "CPU implementer\t: 0x61\nCPU part\t: 0x022\n"
    assert bench.parse_cpu_model(other, "aarch64") == "aarch64 implementer 0x61 part 0x22"
    assert bench.parse_cpu_model("", "aarch64") == "aarch64"
    assert isinstance(bench.host_cpu_model(), str) and bench.host_cpu_model()


def test_accuracy_record_against_the_oracle_rows():
    ref = np.zeros((3, 2, 4))
    ref[1] = 1.0
    gpu = np.zeros((5, 2, 4), dtype=np.float32)
    gpu[2] = 1.0 + 2 ** -8      # row 2 of the batch is the second checked row
    gpu[0, 0, 0] = 0.5
    acc = bench.accuracy_vs_oracle(gpu, ref, [0, 2, 4])
    assert acc["max_abs_err"] == 0.5
    assert abs(acc["mean_abs_err"] - (0.5 + 8 * 2 ** -8) / 24) < 1e-12
    assert acc["max_abs_ref"] == 1.0 and acc["nonfinite"] == 0
    assert acc["rows_checked"] == 3 and acc["elements_checked"] == 24
    gpu[4, 1, 3] = np.nan
    acc = bench.accuracy_vs_oracle(gpu, ref, [0, 2, 4])
    assert acc["nonfinite"] == 1 and acc["max_abs_err"] == 0.5
    json.dumps(acc, allow_nan=False)  # no NaN or inf reaches the JSON line


def test_nvtx_range_never_fails():
    with bench.nvtx_range("region"):
        pass
