"""Measures the tensor-core decode's key-block count on this GPU and writes the table the
planner reads (csrc/decode_blocks_table.h).

    python -m scaled_dot_product_nv_gb300.tune_decode_blocks measure OUT.jsonl
    python -m scaled_dot_product_nv_gb300.tune_decode_blocks table OUT.jsonl [MORE.jsonl ...]

`measure` times every candidate block count (forced through NV_SDPA_DECODE_BLOCKS) on the
decode grid of the pages ("nuvec-core 0.6.1 tests/attention_plan.rs", grid(): keys
1023 ... 65537, heads (32,4,128), (16,2,256), (24,2,128), (8,1,64)), with one and with
eight sequences and 1, 4 or 8 queries each, in f16, as CUDA-graph replays of 20 calls
whose keys and values rotate through more than three L2 sizes of memory (so only HBM
reads and device time count).  `table` picks, for each head bucket, work units per
batch item (KV heads x 16-row tiles) and span of keys, the block count whose eight-
sequence rate is within 5 % of the best measured there and which, among those, has the
best geometric mean of the two batch sizes' rates relative to their bests (the split
may not depend on the batch size: a batch item must get the bits it gets alone).
"""
from __future__ import annotations

import json
import math
import os
import sys
from collections import defaultdict

HEADS = [(32, 4, 128), (16, 2, 256), (24, 2, 128), (8, 1, 64)]
LKS = [1023, 1024, 4096, 8192, 8193, 32769, 65537]
LQS = [1, 4, 8]
BATCHES = [1, 8]
COARSE = [1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 96, 128, 192, 256]
LARGE_BATCH_FLOOR = 0.95
HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(HERE, "csrc", "decode_blocks_table.h")


def units_per_item(hq, hkv, lq):
    g = hq // hkv
    return hkv * (-(-(g * lq) // 16))


def measure(path):
    import torch
    import scaled_dot_product_nv_gb300 as nv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = 129 * 2 ** 20
    pool_elems = (3 * l2) // 2 + (1 << 20)
    pool = torch.randn(pool_elems, device=dev, dtype=torch.float16) * 0.5
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    with open(path, "w") as out:
        for (hq, hkv, d) in HEADS:
            for lk in LKS:
                for B in BATCHES:
                    n_kv = B * hkv * lk * d
                    kv_bytes = 4 * n_kv
                    per = (2 * n_kv + 255) // 256 * 256
                    if per > pool_elems:
                        big = torch.randn(2 * n_kv, device=dev, dtype=torch.float16) * 0.5
                        sets = [(big[:n_kv].view(B, hkv, lk, d), big[n_kv:].view(B, hkv, lk, d))]
                    else:
                        sets = [(pool[s * per:s * per + n_kv].view(B, hkv, lk, d),
                                 pool[s * per + n_kv:s * per + 2 * n_kv].view(B, hkv, lk, d))
                                for s in range(min(pool_elems // per, 4096))]
                    for lq in LQS:
                        q = torch.randn(B, hq, lq, d, device=dev, dtype=torch.float16)
                        o = torch.empty(B, hq, lq, d, device=dev, dtype=torch.float16)
                        lse = torch.empty(B, hq, lq, device=dev, dtype=torch.float32)
                        sk = torch.randn(hq, device=dev, dtype=torch.float16)
                        dims = (B, hq, hkv, lq, lk, d, d)
                        units = units_per_item(hq, hkv, lq)
                        slots = sms * (8 if d <= 128 else 3)
                        s8 = max(1, slots // (8 * units))
                        cands = set(COARSE)
                        if lk >= 8192:
                            cands |= {k * s8 for k in range(1, 13)} | {k * s8 - 1 for k in range(2, 13)}
                        for nb in sorted(c for c in cands if c <= min(1024, -(-lk // 64))):
                            os.environ["NV_SDPA_DECODE_BLOCKS"] = str(nb)
                            st, pl = nv.nv_sdpa_plan(dims, 1, 1, 1)
                            if st != 0 or pl["kernel"] != "decode_mma":
                                continue
                            n = 20
                            side = torch.cuda.Stream()

                            def calls(cs, base):
                                for i in range(n):
                                    k, v = sets[(base + i) % len(sets)]
                                    r = nv.nv_sdpa(q.data_ptr(), k.data_ptr(), v.data_ptr(), dims, 1, 0,
                                                   sk.data_ptr(), d ** -0.5, o.data_ptr(), lse.data_ptr(), 1, cs)
                                    if r != 0:
                                        raise nv.NvSdpaError(r)
                            side.wait_stream(torch.cuda.current_stream())
                            with torch.cuda.stream(side):
                                calls(side.cuda_stream, 0)
                            torch.cuda.current_stream().wait_stream(side)
                            torch.cuda.synchronize()
                            g = torch.cuda.CUDAGraph()
                            with torch.cuda.graph(g, stream=side):
                                calls(side.cuda_stream, n)
                            g.replay()
                            torch.cuda.synchronize()
                            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                            a.record()
                            for _ in range(3):
                                g.replay()
                            b.record()
                            torch.cuda.synchronize()
                            ms = a.elapsed_time(b) / (3 * n)
                            out.write(json.dumps(dict(hq=hq, hkv=hkv, d=d, lk=lk, B=B, lq=lq, nblk=pl["nblk"],
                                                      kpb=pl["keys_per_blk"], ms=ms,
                                                      gbs=kv_bytes / ms / 1e6)) + "\n")
                        os.environ.pop("NV_SDPA_DECODE_BLOCKS", None)
                    del sets


def select(paths):
    """The table entries [(dmax, units, span, nblk, kpb, score)] from measurement files."""
    cells = defaultdict(lambda: defaultdict(dict))
    kpb_of = {}
    for p in paths:
        for line in open(p):
            r = json.loads(line)
            if "gbs" not in r or r.get("planner"):
                continue
            key = (max(r["d"], r["d"]), units_per_item(r["hq"], r["hkv"], r["lq"]), r["lk"])
            cell = cells[key][((r["hq"], r["hkv"], r["lq"]), r["B"])]
            cell[r["nblk"]] = max(r["gbs"], cell.get(r["nblk"], 0.0))
            kpb_of[(r["lk"], r["nblk"])] = r["kpb"]
    gm = lambda xs: math.exp(sum(math.log(x) for x in xs) / len(xs))
    table = []
    for key in sorted(cells):
        runs = cells[key]
        common = sorted(set.intersection(*[set(v) for v in runs.values()]))
        large = [nb for nb in common
                 if all(v[nb] >= LARGE_BATCH_FLOOR * max(v.values()) for (c, B), v in runs.items() if B == 8)]
        score = lambda nb: gm([v[nb] / max(v.values()) for v in runs.values()])
        nb = max(large or common, key=score)
        table.append((key[0], key[1], key[2], nb, kpb_of[(key[2], nb)], round(score(nb), 3)))
    return table


def write_header(table, sources):
    lines = [
        "// Generated by scaled_dot_product_nv_gb300/tune_decode_blocks.py from measurements on a GB300",
        "// (" + ", ".join(os.path.basename(s) for s in sources) + ").  Do not edit by hand.",
        "//",
        "// The key blocks of the tensor-core decode: for a head bucket (max(d, dv)), work units per",
        "// batch item (KV heads x 16-row tiles) and span of keys, the keys per block whose",
        "// eight-sequence rate was within 5 % of the best measured and which, among those, best",
        "// balanced the one- and eight-sequence rates.  The planner takes the nearest entry and",
        "// cuts the call's span into blocks of its keys_per_blk.",
        "#pragma once",
        "",
        "#include <stdint.h>",
        "",
        "namespace nvsdpa {",
        "",
        "struct DecodeBlocksEntry {",
        "  int32_t dmax, units, span, nblk, keys_per_blk;",
        "};",
        "",
        "constexpr DecodeBlocksEntry kDecodeBlocks[] = {",
    ]
    for dmax, units, span, nb, kpb, score in table:
        lines.append(f"    {{{dmax}, {units}, {span}, {nb}, {kpb}}},  // balance {score}")
    lines += ["};", "", "}  // namespace nvsdpa", ""]
    with open(HEADER, "w") as f:
        f.write("\n".join(lines))


def main(argv):
    if len(argv) >= 2 and argv[0] == "measure":
        measure(argv[1])
    elif len(argv) >= 2 and argv[0] == "table":
        write_header(select(argv[1:]), argv[1:])
    else:
        print(__doc__)
        return 2
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
