"""Run one GEMM shape on the GPU through the C ABI: a driver for profilers and sweeps.

    python -m dense_gemm_blackwell_02_gb300.run M N K [--in f16|bf16] [--out f16|bf16|f32]
                                                [--reps R] [--config JSON]

Operands are drawn on the device (uniform [-1, 1], fixed seed), then `gemm_run` is
called R times on one stream.  Prints the kernel configuration the library chose and
the device status word; exits non-zero if a launch or the status reports an error.
"""
from __future__ import annotations

import argparse
import json
import sys

import torch

from .binding import Gemm

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("M", type=int)
    ap.add_argument("N", type=int)
    ap.add_argument("K", type=int)
    ap.add_argument("--in", dest="din", default="f16", choices=["f16", "bf16"])
    ap.add_argument("--out", dest="dout", default="f16", choices=sorted(DTYPES))
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--config", default=None, help="JSON gemm_config_t fields")
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    A = (torch.rand(a.M, a.K, generator=gen, device=dev) * 2 - 1).to(DTYPES[a.din])
    B = (torch.rand(a.N, a.K, generator=gen, device=dev) * 2 - 1).to(DTYPES[a.din])
    C = torch.empty(a.M, a.N, dtype=DTYPES[a.dout], device=dev)
    with Gemm() as g:
        if a.config:
            g.set_config(**json.loads(a.config))
        for _ in range(a.reps):
            g.run(A, B, C)
        torch.cuda.synchronize()
        code, word = g.device_status()
        print(json.dumps({"M": a.M, "N": a.N, "K": a.K, "kernel": g.last_config(),
                          "status": code, "status_word": word}))
    return 1 if code else 0


if __name__ == "__main__":
    sys.exit(main())
