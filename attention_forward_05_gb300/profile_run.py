"""Runs one kernel family on a named synthetic workload a few times (for profilers such as ncu).

    python -m attention_forward_05_gb300.profile_run --workload mh_prefill --launches 2
    python -m attention_forward_05_gb300.profile_run --workload decode --B 4 --launches 2
    python -m attention_forward_05_gb300.profile_run --workload mh_prefill --bwd --launches 2
    python -m attention_forward_05_gb300.profile_run --workload decode --B 8 --hkv 4 --launches 2

The first launch is a warm-up; the process exits 0 after a device synchronise
and a device-error check.  --B / --H override the workload's batch and heads
(keeping the per-head shapes) so that a capture can stay small.  --hkv N runs the
decode workload as grouped-query decode (fa_decode_splitkv_gqa) with N key/value
heads shared by its query heads.
"""
from __future__ import annotations

import argparse
import dataclasses
import sys

import torch

import attention_forward_05_gb300 as fa
from attention_forward_05_gb300 import accounting
from attention_forward_05_gb300.inputs import WORKLOADS, make_dout, make_qkv, merge_order, workload_inputs


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=sorted(WORKLOADS), required=True)
    ap.add_argument("--launches", type=int, default=2)
    ap.add_argument("--B", type=int, default=0)
    ap.add_argument("--H", type=int, default=0)
    ap.add_argument("--time", action="store_true", help="time the launches with CUDA events and print the rate")
    ap.add_argument("--causal", action="store_true", help="causal mask (prefill workloads)")
    ap.add_argument("--bwd", action="store_true", help="time the backward (fa_bwd) after one forward (prefill)")
    ap.add_argument("--hkv", type=int, default=0, help="decode: grouped-query decode with this many key/value heads")
    a = ap.parse_args(argv)
    w = WORKLOADS[a.workload]
    if a.B:
        w = dataclasses.replace(w, B=a.B)
    if a.H:
        w = dataclasses.replace(w, H=a.H)
    dev = torch.device("cuda:0")
    q, k, v = workload_inputs(w, device=dev)
    if a.hkv:
        if not w.splits or w.H % a.hkv:
            ap.error("--hkv takes the decode workload and a divisor of its head count")
        _, k, v = make_qkv(w.B, a.hkv, 1, w.Nk, w.d, w.dtype, seed=w.seed + a.hkv, device=dev)
    order = torch.as_tensor(merge_order(w.splits, w.order_seed), device=dev) if w.splits else None
    o = torch.empty_like(q) if not w.splits else None
    lse = torch.empty((w.B, w.H, w.Nq), device=dev) if not w.splits else None

    if a.bwd:
        if w.splits:
            ap.error("--bwd takes a prefill workload")
        dout = make_dout(w.B, w.H, w.Nq, w.d, w.dtype, seed=w.seed + 700, device=dev)
        fa.fa_fwd(q, k, v, scale=w.scale, o=o, lse=lse, causal=a.causal)
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.Nq, w.d), dtype=torch.uint8, device=dev)

    def run():
        if a.bwd:
            fa.fa_bwd(q, k, v, o, dout, lse, scale=w.scale, causal=a.causal, dq=grads[0], dk=grads[1], dv=grads[2],
                      workspace=ws)
        elif a.hkv:
            fa.fa_decode_splitkv_gqa(q, k, v, w.splits, merge_order=order)
        elif w.splits:
            fa.fa_decode_splitkv_ex(q, k, v, w.splits, merge_order=order)
        else:
            fa.fa_fwd(q, k, v, scale=w.scale, o=o, lse=lse, causal=a.causal)

    torch.cuda.synchronize()
    run()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(a.launches):
        run()
    end.record()
    torch.cuda.synchronize()
    if a.time and a.launches:
        ms = start.elapsed_time(end) / a.launches
        if a.bwd:
            fl = accounting.bwd_flops_causal(w.B, w.H, w.Nq, w.Nk, w.d) if a.causal else \
                accounting.bwd_flops(w.B, w.H, w.Nq, w.Nk, w.d)
            rate = f"{fl / ms / 1e9:.1f} TFLOP/s (backward{', causal' if a.causal else ''})"
        elif a.hkv:
            rate = f"{accounting.decode_gqa_min_bytes(w.B, w.H, a.hkv, w.Nk, w.d) / ms / 1e6:.1f} GB/s"
        elif w.splits:
            rate = f"{accounting.decode_min_bytes(w.B, w.H, w.Nk, w.d) / ms / 1e6:.1f} GB/s"
        elif a.causal:
            rate = f"{accounting.fwd_flops_causal(w.B, w.H, w.Nq, w.Nk, w.d) / ms / 1e9:.1f} TFLOP/s (causal)"
        else:
            rate = f"{accounting.fwd_flops(w.B, w.H, w.Nq, w.Nk, w.d) / ms / 1e9:.1f} TFLOP/s"
        print(f"time: {w.name} {ms * 1e3:.1f} us/launch {rate}")
    if fa.fa_check_device_error() != fa.FA_OK:
        print("device timeout", file=sys.stderr)
        return 1
    hkv = f" Hkv={a.hkv}" if a.hkv else ""
    print(f"ok: {w.name} B={w.B} H={w.H}{hkv} Nq={w.Nq} Nk={w.Nk} d={w.d} launches={a.launches}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
