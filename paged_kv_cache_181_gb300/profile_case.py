"""Run a few forwards of one workload for a profiler to capture.

    python -m paged_kv_cache_181_gb300.profile_case --workload long-window-40L-bf16 --layers 1 --steps 3

Builds the workload's pools and metadata like the benchmark does (with
``--layers`` layers instead of the workload's own count, to keep a capture
small), runs ``--steps`` forwards -- each layer: KV write, then paged
attention -- and checks the device error word.  It prints nothing of the
timing: numbers taken under a profiler are not benchmark figures.
"""

from __future__ import annotations

import argparse

import torch

from . import _lib, configs, workload


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="long-window-40L-bf16")
    ap.add_argument("--layers", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--fused", action="store_true", help="paged_kv_write_attn instead of the two calls")
    ap.add_argument("--packed", default=None, help="run this packed batch's attention call instead (configs.PACKED)")
    ap.add_argument("--gather", action="store_true", help="also stage each layer's window (paged_kv_gather)")
    ap.add_argument("--dtype", choices=["f32", "bf16", "f16"], default=None,
                    help="the workload's shapes with this input dtype (f32 runs the CUDA-core kernel)")
    ap.add_argument("--pool-blocks", type=int, default=None,
                    help="blocks per layer pool (default: the workload's); a smaller pool keeps a capture's device "
                         "memory small without changing the blocks the call reads or writes")
    args = ap.parse_args()
    if args.packed:
        from . import packed

        pc = packed.build_packed(configs.PACKED[args.packed], poison=False)
        for _ in range(args.steps):
            pc.attend(flags=args.flags)
        torch.cuda.synchronize()
        bits = _lib.check()
        if bits:
            raise SystemExit(f"device error word 0x{bits:x}")
        print(f"profile_case: {args.packed}, {args.steps} attention call(s): ok")
        return
    import dataclasses

    w = {**configs.ALL, **configs.VARIANTS}[args.workload]
    if args.pool_blocks:
        w = dataclasses.replace(w, pool_blocks=args.pool_blocks)
    if args.dtype:
        w = dataclasses.replace(w, dtype=args.dtype)
    case = workload.build_case(w, device="cuda", layers=args.layers, data_device="cuda")
    st = case.make_staging() if args.gather else None
    for _ in range(args.steps):
        case.step(flags=args.flags, fused=args.fused)
        if st is not None:
            for layer in range(case.layers):
                case.stage(layer, st)
    torch.cuda.synchronize()
    bits = _lib.check()
    if bits:
        raise SystemExit(f"device error word 0x{bits:x}")
    api = "fused" if args.fused else "two calls"
    print(f"profile_case: {w.name}, {args.layers} layer(s), {args.steps} forward(s), {api}: ok")


if __name__ == "__main__":
    main()
