"""Workloads for the bounds-checked build (run as a script by tests/test_gpu_bounds.py with
ZERO_LIBZERO naming libzero_checked.so): every kernel of the step and the gather, each
compared with the oracle, then the build's bounds report. Prints one JSON line."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import sharded_emulated_reduce_gb300 as z  # noqa: E402
from synth import workloads as wl  # noqa: E402

from parity import Runner, h16  # noqa: E402
from test_gpu_gather import run_gather  # noqa: E402


def small(**kw) -> wl.Workload:
    base = dict(name="bounds", cfg=900, n=4099, nd=4, align=8, stage=2, r0=0, r1=4,
                loss_scale=1024.0, grad_sigma=1e-3, clip=1.0, steps=2, m_sigma=1e-3,
                v_sigma=1e-6)
    base.update(kw)
    return wl.Workload(**base)


def main() -> int:
    torch.cuda.set_device(0)
    z.zero_bounds_check(reset=True)
    exact = {}
    cases = {
        # the one-launch step: state in shared memory, then a slice too long for that
        "one launch": small(n=1_000_003),
        "one launch, wide slices": small(n=3_000_001, cfg=901),
        # register-load reduce and the update, with a ragged tail
        "reduce + update": small(n=5_000_003, cfg=902),
        # bulk-load reduce: 16 ranks, 64 ranks (a rank count read at run time: 17)
        "bulk reduce, 16 ranks": small(n=6_000_011, nd=16, r1=16, cfg=903),
        "bulk reduce, 17 ranks": small(n=4_000_037, nd=17, r1=17, cfg=904),
        "bulk reduce, 64 ranks": small(n=4_500_001, nd=64, r1=64, cfg=905, steps=1),
    }
    for name, w in cases.items():
        exact[name] = bool(Runner(w).run().exact)
    # the gather: aligned layers, layers misaligned against the shards, and relative
    # misalignment of source and destination
    n, nd = 3_000_000, 8
    run_gather(n, nd, 8, [0, 1_000_000, 2_000_000, n])
    run_gather(n, nd, 8, [0, 1_000_001, 1_999_997, n])
    run_gather(n, nd, 8, [0, 700_003, n], dst_pad=3, src_pad=1)
    exact["gather"] = True  # run_gather asserts every element against the oracle
    # the allocation-free step
    m = 1_000_000
    g = torch.Generator(device="cuda").manual_seed(7)
    grads = [(torch.randn(m, device="cuda", generator=g) * 1e-3).half() for _ in range(4)]
    master = torch.randn(m, device="cuda", generator=g) * 0.02
    mm, vv = torch.zeros(m, device="cuda"), torch.zeros(m, device="cuda")
    p16 = torch.zeros(m, dtype=torch.float16, device="cuda")
    step = torch.zeros(1, dtype=torch.int64, device="cuda")
    z.zero_shard_step_noalloc(4, m, m, grads, master, mm, vv, p16, step,
                              dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                   weight_decay=0.01), 1.0, 1.0)
    info = z.zero_noalloc_step_result()
    exact["allocation-free step"] = info.status == 0 and int(step.item()) == 1 and bool(
        np.array_equal(h16(p16), h16(master.half())))
    torch.cuda.synchronize()
    rep = z.zero_bounds_check(reset=True)
    # the checks themselves: a range past the end of a buffer is recorded (not accessed)
    z.zero_selftest_bounds()
    probe = z.zero_bounds_check(reset=True)
    print(json.dumps({"exact": exact, **rep, "probe": probe}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
