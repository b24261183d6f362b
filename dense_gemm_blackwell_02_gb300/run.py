"""Run one GEMM shape, or one grouped MoE workload, on the GPU through the C ABI: a
driver for profilers and sweeps.

    python -m dense_gemm_blackwell_02_gb300.run M N K [--in f16|bf16|e4m3|e5m2]
                                                [--out f16|bf16|f32] [--reps R]
                                                [--config JSON] [--blockwise BM]
    python -m dense_gemm_blackwell_02_gb300.run --moe NAME [--experts E] [--reps R]

Operands are drawn on the device (uniform [-1, 1], fixed seed), then `gemm_run` (or,
with --moe, `gemm_run_grouped` over the workload's experts, the first E of them with
--experts; with --blockwise BM and FP8 inputs, `gemm_run_blockwise` with scales in
[2^-3, 2^3] per BM rows of A and 128 of K, and per 128 x 128 of B) is called R times on
one stream.  Prints the kernel configuration the
library chose and the device status word; exits non-zero if a launch or the status
reports an error.
"""
from __future__ import annotations

import argparse
import json
import sys

import torch

from .binding import Gemm

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
          "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _moe_problems(name: str, experts: int, dev, gen):
    import seeded_inputs as si
    wl = si.MOE_WORKLOADS[name]
    counts = si.moe_counts(wl.experts, wl.rows, wl.seed)
    if experts:
        counts = counts[:experts]
    tin, tout = si.TORCH_DTYPE[wl.dtype_in], si.TORCH_DTYPE[wl.dtype_out]
    return [((torch.rand(m, wl.K, generator=gen, device=dev) * 2 - 1).to(tin),
             (torch.rand(wl.N, wl.K, generator=gen, device=dev) * 2 - 1).to(tin),
             torch.empty(m, wl.N, dtype=tout, device=dev)) for m in counts]


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("M", type=int, nargs="?")
    ap.add_argument("N", type=int, nargs="?")
    ap.add_argument("K", type=int, nargs="?")
    ap.add_argument("--in", dest="din", default="f16", choices=["f16", "bf16", "e4m3", "e5m2"])
    ap.add_argument("--out", dest="dout", default="f16", choices=["f16", "bf16", "f32"])
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--config", default=None, help="JSON gemm_config_t fields")
    ap.add_argument("--moe", default=None, help="a grouped MoE workload of seeded_inputs")
    ap.add_argument("--experts", type=int, default=0, help="with --moe: only the first E experts")
    ap.add_argument("--blockwise", type=int, default=0,
                    help="FP8 inputs: block scales, one per BM rows of A and 128 of K")
    a = ap.parse_args(argv)
    if a.moe is None and None in (a.M, a.N, a.K):
        ap.error("M N K are required without --moe")
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    with Gemm() as g:
        if a.config:
            g.set_config(**json.loads(a.config))
        if a.moe:
            probs = _moe_problems(a.moe, a.experts, dev, gen)
            for _ in range(a.reps):
                g.run_grouped(probs)
            shape = {"moe": a.moe, "experts": len(probs), "rows": sum(p[0].shape[0] for p in probs)}
        else:
            A = (torch.rand(a.M, a.K, generator=gen, device=dev) * 2 - 1).to(DTYPES[a.din])
            B = (torch.rand(a.N, a.K, generator=gen, device=dev) * 2 - 1).to(DTYPES[a.din])
            C = torch.empty(a.M, a.N, dtype=DTYPES[a.dout], device=dev)
            if a.blockwise:
                nkb = -(-a.K // 128)
                sfa = torch.exp2(torch.rand(nkb, -(-a.M // a.blockwise), generator=gen, device=dev) * 6 - 3)
                sfb = torch.exp2(torch.rand(nkb, -(-a.N // 128), generator=gen, device=dev) * 6 - 3)
            for _ in range(a.reps):
                if a.blockwise:
                    g.run_blockwise(A, B, C, sfa, sfb, a.blockwise)
                else:
                    g.run(A, B, C)
            shape = {"M": a.M, "N": a.N, "K": a.K, "in": a.din, "out": a.dout,
                     "blockwise": a.blockwise}
        torch.cuda.synchronize()
        code, word = g.device_status()
        print(json.dumps({**shape, "kernel": g.last_config(), "status": code, "status_word": word}))
    return 1 if code else 0


if __name__ == "__main__":
    sys.exit(main())
