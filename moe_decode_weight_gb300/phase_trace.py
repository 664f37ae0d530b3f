"""Phase timelines of the MoE stack kernel (per layer) and the FP8 head, from the profiling build.

``build(trace=True)`` compiles the same kernels with ``-DMDW_TRACE``. Thread 0 of every block
then writes ``%globaltimer`` at fixed points of every layer into a device table
(``mdw_trace_read``). This module runs the stack on synthetic weights (seed 3, the bench's
weights) with that library and prints, per layer, the median and the maximum over blocks of
each phase. A phase runs from the previous point in kernel order to its own point.

Points inside loops (gate/up rounds, pair chunks) keep their last value, so those phases
cover the last round / chunk, and "earlier rounds" / "earlier chunks" hold the rest.
A one-token window builds its routing tables inside the top-k, so "gates" .. "pairs" are ~0
there.

    python -m moe_decode_weight_gb300.phase_trace --layers 8 --m 1
    python -m moe_decode_weight_gb300.phase_trace --head --m 1

The product library ``libmdw.so`` is neither rebuilt nor loaded.
"""

from __future__ import annotations

import argparse
import ctypes as C

import numpy as np

TRACE_LAYERS, TRACE_POINTS, TRACE_BLOCKS = 64, 24, 256   # the device table's shape

# (point id, name of the phase that ends there), in kernel order; point 0 starts a layer
PHASES = [
    (12, "residual poll"),       # up to two tokens in a stack: r_l from the tagged words (~0 else)
    (1, "input"),                # r -> bf16 x (stack: RMSNorm) -> E4M3 x-hat
    (2, "router rows"),          # router rows published as tagged words (M > 16: x-hat codes)
    (3, "logit poll"),           # (top-k warp 0; imposed routing: ~0, its wait is in "top-k rank")
    (4, "top-k threshold"),      # lane bests, bitonic sort, the K-th best
    (10, "top-k rank"),          # candidates compacted and ranked
    (20, "gates"),               # more than one token: softmax of the selected logits
    (21, "union scan"),          # expert bitmap and its prefix counts
    (11, "slots"),               # the union's slots (one token: all tables, in registers)
    (22, "pairs"),               # token masks, slot offsets, the pair lists
    (5, "gate/up list"),
    (15, "gate/up earlier rounds"),
    (16, "gate/up last round"),
    (6, "SwiGLU+arrive"),
    (7, "B2 wait"),              # W2 prefetch and the first down unit list run in the wait
    (17, "down earlier chunks"),
    (18, "h quantisation"),
    (13, "down unit list"),
    (19, "down units"),
    (14, "leftover rows+sum"),
    (8, "output"),
    (9, "B3"),                   # no residual barrier up to two tokens (~0 there)
]


def summarise(tr: np.ndarray):
    """tr: [layers][TRACE_POINTS][blocks] nanosecond stamps. Returns one dict per layer:
    {"total_us": first start to last B3 exit, phase name: (median_us, max_us) over blocks}."""
    out = []
    for lay in tr.astype(np.float64):
        row = {"total_us": float((lay[9].max() - lay[0].min()) / 1000.0)}
        prev = 0
        for point, name in PHASES:
            d = (lay[point] - lay[prev]) / 1000.0
            row[name] = (float(np.median(d)), float(d.max()))
            prev = point
        out.append(row)
    return out


HEAD_SLOTS, HEAD_WARPS = 24, 12    # per-block slots of the head's table; warp w stamps slot 8 + w
# (slot, name of the per-block phase that ends there), in kernel order from slot 0
HEAD_PHASES = [(1, "hidden states"), (2, "tiles"), (20, "cut tiles"), (21, "warp lists"),
               (22, "block tree"), (3, "block list out")]


def summarise_head(tr: np.ndarray):
    """tr: [blocks][HEAD_SLOTS] nanosecond stamps of one head launch (group / final slots
    older than this launch's first start are stale and ignored). Returns per-block phases
    (min, median, max over blocks, µs) and the launch's timeline from its first start."""
    tr = tr.astype(np.float64)
    t0 = tr[:, 0].min()
    out = {}
    prev = 0
    for slot, name in HEAD_PHASES:
        d = (tr[:, slot] - tr[:, prev]) / 1000.0
        out[name] = (float(d.min()), float(np.median(d)), float(d.max()))
        prev = slot
    warps = tr[:, 8:8 + HEAD_WARPS]
    spread = (warps.max(axis=1) - warps.min(axis=1)) / 1000.0
    out["warp spread"] = (float(spread.min()), float(np.median(spread)), float(spread.max()))
    done = (tr[:, 2] - t0) / 1000.0
    out["tiles done (from start)"] = (float(done.min()), float(np.median(done)), float(done.max()))
    grp = tr[:, 4] >= t0
    fin = tr[:, 5] >= t0
    out["group mergers"] = int(grp.sum())
    out["group merge start"] = float(np.median(tr[grp, 4] - t0) / 1000.0) if grp.any() else None
    if fin.any():
        b = int(np.argmax(np.where(fin, tr[:, 5], 0.0)))
        out["final merge start"] = float((tr[b, 5] - t0) / 1000.0)
        out["end"] = float((tr[b, 6] - t0) / 1000.0)
    return out


def format_head(summary) -> str:
    lines = ["head, per block: min / median / max (us)"]
    for key, v in summary.items():
        if isinstance(v, tuple):
            lines.append(f"  {key}: {v[0]:.2f} / {v[1]:.2f} / {v[2]:.2f}")
        elif v is not None:
            lines.append(f"  {key}: {v:.2f}" if isinstance(v, float) else f"  {key}: {v}")
    return "\n".join(lines)


def format_rows(rows) -> str:
    lines = ["per layer: phase median / max over blocks (us), from the previous point"]
    for l, row in enumerate(rows):
        parts = [f"{name} {row[name][0]:.2f}/{row[name][1]:.2f}" for _, name in PHASES]
        lines.append(f"L{l}: total {row['total_us']:.2f} | " + " | ".join(parts))
    return "\n".join(lines)


def main() -> None:
    import torch

    from moe_decode_weight_gb300 import api, build, synth

    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--m", type=int, default=1)
    ap.add_argument("--runs", type=int, default=4, help="launches; the last one is reported")
    ap.add_argument("--head", action="store_true",
                    help="trace the FP8 head over the full vocabulary instead of the MoE stack")
    args = ap.parse_args()
    if args.head:
        return head_main(args)
    L, M = args.layers, args.m
    if not 1 <= L <= TRACE_LAYERS:
        raise SystemExit(f"--layers must be 1..{TRACE_LAYERS}")
    api.LIB_PATH = build.build(trace=True)
    api._lib = None
    dev = torch.device("cuda:0")
    layers = []
    for l in range(L):
        (w13q, w13s, w2q, w2s), sh = synth.layer_experts(3, l, synth.NUM_EXPERTS, device=dev)
        wr = synth.router_weight(3, l, synth.NUM_EXPERTS).to(dev)
        layers.append(api.MoeWeights(wr, w13q, w13s, w2q, w2s, tuple(sh), synth.TOP_K))
    arr = api._layer_array(layers)
    ws = torch.zeros(api.mdw_stack_workspace_bytes(layers, None, M, 1), dtype=torch.uint8, device=dev)
    resid = torch.zeros((L + 1, M, synth.HIDDEN), dtype=torch.bfloat16, device=dev)
    for it in range(args.runs):
        r0 = synth.hidden_states(3, M, 100 + it).to(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        api.moe_decode_stack(arr, None, r0, None, ws, resid_out=resid)
        e1.record()
        torch.cuda.synchronize()
        print(f"run {it}: {e0.elapsed_time(e1) * 1000.0:.1f} us, status {api.mdw_device_status(ws)}")
    lib = api.lib()
    lib.mdw_trace_read.argtypes = [C.c_void_p, C.c_size_t]
    buf = np.zeros(TRACE_LAYERS * TRACE_POINTS * TRACE_BLOCKS, dtype=np.uint64)
    if lib.mdw_trace_read(buf.ctypes.data, buf.nbytes) != 0:
        raise SystemExit("mdw_trace_read failed")
    G = torch.cuda.get_device_properties(0).multi_processor_count
    tr = buf.reshape(TRACE_LAYERS, TRACE_POINTS, TRACE_BLOCKS)[:L, :, :G]
    print(f"M = {M}, {L} layers, {G} blocks")
    print(format_rows(summarise(tr)))


def head_main(args) -> None:
    import torch

    from moe_decode_weight_gb300 import api, build, synth

    M = args.m
    api.LIB_PATH = build.build(trace=True)
    api._lib = None
    dev = torch.device("cuda:0")
    w = synth.lm_head_weight(1, synth.VOCAB).to(dev)
    q = torch.empty((synth.VOCAB, synth.HIDDEN), dtype=torch.uint8, device=dev)
    sc = torch.empty(synth.VOCAB, dtype=torch.float32, device=dev)
    head = api.quantize_lm_head_fp8(w, q, sc)
    del w
    h = synth.hidden_states(1, M, 0).to(dev)
    ws = torch.zeros(api.mdw_lm_head_workspace_bytes(head, M, synth.TOPK_VOCAB), dtype=torch.uint8, device=dev)
    am = torch.zeros(M, dtype=torch.int32, device=dev)
    for it in range(args.runs):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        api.lm_head_fp8(head, h, am, ws, topk=synth.TOPK_VOCAB)
        e1.record()
        torch.cuda.synchronize()
        print(f"run {it}: {e0.elapsed_time(e1) * 1000.0:.1f} us, status {api.mdw_device_status(ws)}")
    lib = api.lib()
    lib.mdw_head_trace_read.argtypes = [C.c_void_p, C.c_size_t]
    buf = np.zeros(TRACE_BLOCKS * HEAD_SLOTS, dtype=np.uint64)
    if lib.mdw_head_trace_read(buf.ctypes.data, buf.nbytes) != 0:
        raise SystemExit("mdw_head_trace_read failed")
    G = min(torch.cuda.get_device_properties(0).multi_processor_count, TRACE_BLOCKS)
    print(f"FP8 head, M = {M}, {G} blocks" + (" (the last of several 16-token launches)" if M > 16 else ""))
    print(format_head(summarise_head(buf.reshape(TRACE_BLOCKS, HEAD_SLOTS)[:G])))


if __name__ == "__main__":
    main()
