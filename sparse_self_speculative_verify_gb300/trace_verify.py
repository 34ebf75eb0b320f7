"""Timeline of the tensor-core verify kernel: where a verify call's time goes.

Builds the diagnostic variant of the library (``build(variant="trace")``: the same kernels, plus a
per-block record of global-timer and SM-cycle stamps) into its own directory, loads it in place of
the library proper for this process, runs ``ssd_verify_attn`` on a seeded workload a few times
(L2 flushed before each call) and breaks the last launch down:

* ramp: cycles from a block's entry to the start of its first item's tiles;
* steady rate: cycles per 128-token tile of K and V, from consecutive items of the same block
  (the time between two items' epilogues against their tile counts);
* per-item cost: the intercept of that fit, the time an item costs beyond its tiles;
* tail: the spread of the blocks' exit times.

Usage: ``python -m sparse_self_speculative_verify_gb300.trace_verify [workload] [--dump FILE.npz] [--select]``
with workload qwen3_8b (default), b128_l8k or qwen3_14b_unified (its verify-phase requests).  Prints
a JSON line.  ``--select`` traces ``ssd_verify_select`` instead, as the benchmark's round calls it
(its criticality pass's phases go into the dump).  ``--dump`` also saves the raw per-block, per-tile, masked-tile,
epilogue, producer and softmax-stage records and the requests' lengths.
"""

from __future__ import annotations

import ctypes
import json
import math
import statistics
import sys

import numpy as np
import torch

from . import binding as Bd
from . import build as libbuild
from . import workloads as W

SLOTS, BLOCKS, ITEMS, TILES, MASKED = 128, 256, 40, 256, 16


def run(name: str = "qwen3_8b", dump: str | None = None, select: bool = False) -> dict:
    L = Bd.load(libbuild.build(variant="trace"), as_default=True)
    L.ssd_verify_trace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    L.ssd_verify_trace.restype = ctypes.c_int
    dev = torch.device("cuda", 0)
    spec = W.SPECS[name]
    w = W.make_workload(spec, seed=W.spec_seed(name), device=dev)
    kv = Bd.KVCache.from_workload(w)
    q = w.q_verify
    if w.phase is not None:  # the verify-phase requests of a mixed batch
        vi = torch.nonzero(w.phase == 1).flatten()
        kv = Bd.KVCache(kv.pool, kv.page_table[vi].contiguous(), kv.seq_lens[vi].contiguous(), kv.max_seq_len)
        q = q[vi].contiguous()
    scale = 1.0 / math.sqrt(spec.d)
    ws = Bd.Workspace()
    flush = W.flush_buffer(dev)
    ks, k_max = w.k_per_req, int(w.k_per_req.max())
    for _ in range(4):
        flush.fill_(1.0)
        if select:
            Bd.ssd_verify_select(kv, q, spec.n_cand, scale, ks, k_max, workspace=ws)
        else:
            Bd.ssd_verify_attn(kv, q, spec.n_cand, scale, workspace=ws)
    torch.cuda.synchronize()
    assert Bd.ssd_status() == 0
    tr = np.zeros(BLOCKS * SLOTS, np.uint64)
    assert L.ssd_verify_trace(tr.ctypes.data, tr.nbytes) == 0
    nb = torch.cuda.get_device_properties(0).multi_processor_count
    tr = tr.reshape(BLOCKS, SLOTS).astype(np.int64)[:nb]
    if dump:
        L.ssd_verify_tile_trace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
        L.ssd_verify_tile_trace.restype = ctypes.c_int
        tt = np.zeros(BLOCKS * TILES * 12, np.uint32)
        assert L.ssd_verify_tile_trace(tt.ctypes.data, tt.nbytes) == 0
        L.ssd_verify_masked_trace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
        L.ssd_verify_masked_trace.restype = ctypes.c_int
        tm = np.zeros(BLOCKS * MASKED * 8, np.uint32)
        assert L.ssd_verify_masked_trace(tm.ctypes.data, tm.nbytes) == 0
        L.ssd_verify_epi_trace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
        L.ssd_verify_epi_trace.restype = ctypes.c_int
        te = np.zeros(BLOCKS * ITEMS * 4, np.uint32)
        assert L.ssd_verify_epi_trace(te.ctypes.data, te.nbytes) == 0
        L.ssd_verify_prod_trace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
        L.ssd_verify_prod_trace.restype = ctypes.c_int
        tp = np.zeros(BLOCKS * ITEMS * 4, np.uint32)
        assert L.ssd_verify_prod_trace(tp.ctypes.data, tp.nbytes) == 0
        L.ssd_verify_stage_trace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
        L.ssd_verify_stage_trace.restype = ctypes.c_int
        ts = np.zeros(BLOCKS * 64 * 8, np.uint32)
        assert L.ssd_verify_stage_trace(ts.ctypes.data, ts.nbytes) == 0
        cs = np.zeros(4096 * 16, np.uint64)
        if select:
            L.ssd_crit_select_trace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
            L.ssd_crit_select_trace.restype = ctypes.c_int
            assert L.ssd_crit_select_trace(cs.ctypes.data, cs.nbytes) == 0
        np.savez(dump, trace=tr, producer=tp.reshape(BLOCKS, ITEMS, 4)[:nb], stage=ts.reshape(BLOCKS, 64, 8)[:nb],
                 crit_select=cs.reshape(4096, 16)[:kv.batch * kv.h_kv], tiles=tt.reshape(BLOCKS, TILES, 12)[:nb], masked=tm.reshape(BLOCKS, MASKED, 8)[:nb],
                 epilogue=te.reshape(BLOCKS, ITEMS, 4)[:nb],
                 seq_lens=kv.seq_lens.cpu().numpy(), h_kv=spec.h_kv, n_cand=spec.n_cand)
    entry, exit_, t0 = tr[:, 0], tr[:, 2], int(tr[:, 0].min())
    span_us = (exit_.max() - t0) / 1e3
    mhz = float(np.median(tr[:, 127] / np.maximum(exit_ - entry, 1) * 1e3))  # cycles per us
    tiles, items, first, x, y = 0, 0, [], [], []
    for b in range(nb):
        n = min(int(tr[b, 3]), ITEMS)
        items += n
        prev = None
        for j in range(n):
            st, pk, dn = int(tr[b, 4 + 3 * j]), int(tr[b, 5 + 3 * j]), int(tr[b, 6 + 3 * j])
            nt = pk & 0xFFFFFFFF
            tiles += nt
            if j == 0:
                first.append(st)
            if prev is not None:
                x.append(nt)
                y.append(dn - prev)
            prev = dn
    a_fit, c_fit = np.polyfit(np.array(x, float), np.array(y, float), 1) if len(set(x)) > 1 else (
        statistics.median(np.array(y) / np.array(x)), 0.0)
    exits = (exit_ - t0) / 1e3
    res = {
        "workload": name, "blocks": int(nb), "items": items, "tiles": tiles,
        "kernel_span_us": round(span_us, 1), "sm_mhz": round(mhz, 0),
        "ramp_us": round(statistics.median(first) / mhz, 2),
        "prologue_us": round(float(np.median(tr[:, 1])) / mhz, 2),
        "cycles_per_tile": round(float(a_fit), 0), "cycles_per_item_beyond_tiles": round(float(c_fit), 0),
        "exit_us": {"min": round(float(exits.min()), 1), "median": round(float(np.median(exits)), 1),
                    "max": round(float(exits.max()), 1)},
        "tile_time_per_block_us": round(tiles / nb * a_fit / mhz, 1),
        "item_cost_per_block_us": round(items / nb * c_fit / mhz, 1),
    }
    return res


if __name__ == "__main__":
    args = sys.argv[1:]
    out = None
    sel = "--select" in args
    if sel:
        args.remove("--select")
    if "--dump" in args:
        i = args.index("--dump")
        out = args[i + 1]
        del args[i:i + 2]
    print(json.dumps(run(args[0] if args else "qwen3_8b", out, sel)))
