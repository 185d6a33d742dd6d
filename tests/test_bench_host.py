"""Host-side pieces of bench.py, on the CPU.

* `committed_traffic`: the DRAM figure of a workload is reported only while
  the SHA-256 of its kernel's sources matches the one recorded beside it in
  `profiles/traffic.json`; any other source set (a changed kernel) gives none.
* `packed_device`: the end-to-end loop moves a step's inputs (or results) as
  one copy, so every tensor is rebound to a 256-byte aligned view of one byte
  buffer (contents not carried over), and writes through either side are
  seen by the other.
* the reference arm (`--impl reference`): the fp64 oracle timed on the host
  cores prints one JSON line with the base contract's keys."""
import json
import os
import subprocess
import sys

import torch

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_committed_traffic_follows_the_source_hash():
    table = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert table
    for name, entry in table.items():
        decode = entry["kernel"].startswith("decode_kernel")
        own = bench.DECODE_SOURCES if decode else bench.ATTN_TC_SOURCES
        other = bench.ATTN_TC_SOURCES if decode else bench.DECODE_SOURCES
        assert bench.committed_traffic(name, own) == float(entry["dram_bytes_per_launch"]), name
        assert entry["dram_bytes_per_launch"] == entry["dram_bytes_read"] + entry["dram_bytes_write"]
        assert bench.committed_traffic(name, other) is None, name
    assert bench.committed_traffic("no_such_workload", bench.ATTN_TC_SOURCES) is None


def test_packed_device_rebinds_tensors_to_one_buffer():
    ts = [torch.zeros(3, 5, dtype=torch.int32), torch.zeros(7, dtype=torch.bfloat16),
          torch.zeros(2, 2, 2, dtype=torch.float32), torch.zeros(1, dtype=torch.int64)]
    shapes = [t.shape for t in ts]
    buf, offs = bench.packed_device(ts, torch.device("cpu"))
    assert buf.dtype == torch.uint8
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs) and len(set(offs)) == len(offs)
    base = buf.untyped_storage().data_ptr()
    for t, o, sh in zip(ts, offs, shapes):
        assert t.shape == sh and t.is_contiguous()
        assert t.data_ptr() == base + o
        assert o + t.numel() * t.element_size() <= buf.numel()
    # the contents are not carried over (the buffer is fresh); a write through
    # the buffer is seen by the tensor and the other way round, and no other
    # tensor overlaps either
    buf.zero_()
    ts[0].fill_(7)
    assert (buf[offs[0]:offs[0] + 60].view(torch.int32) == 7).all()
    buf[offs[2]:offs[2] + 32].view(torch.float32).fill_(1.5)
    assert (ts[2] == 1.5).all()
    assert (ts[1] == 0).all() and (ts[3] == 0).all()


def test_reference_arm_prints_one_oracle_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_decode", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.WORKLOAD_META["tiny_decode"]["metric"]
    assert line["unit"] == "GB/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["dtype"] == "f64" and line["config"]["workload"] == "tiny_decode"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
