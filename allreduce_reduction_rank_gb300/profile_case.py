"""Run one allreduce case a few times on cuda:0, for profiling one kernel.

    python -m allreduce_reduction_rank_gb300.profile_case CASE NRANKS BYTES_PER_RANK DTYPE [--calls K]

CASE is one of rsag, rsag_two_phase, ll_allpair (sar_allreduce with that
algorithm), ll (sar_allreduce_ll), ll_fused, ll_cluster,
ll_writeback_multi_dest, ll_writeback_own_output.  The inputs are seeded normal values on the device
(their values do not matter for timing), the buffers are allocated once, and
the case runs K times (default 3) with epochs 1..K, then synchronises and
checks that every output equals the rsag allreduce of the same inputs.  Only
the library's kernels (and torch's initialisation of the inputs) run, so a
profiler filtered on a kernel name sees one launch per call.
"""
from __future__ import annotations

import argparse

import torch

import allreduce_reduction_rank_gb300 as sar

CASES = ("rsag", "rsag_two_phase", "ll_allpair", "ll", "ll_fused", "ll_cluster", "ll_writeback_multi_dest",
         "ll_writeback_own_output")
STORAGE = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32, "e4m3fn": torch.uint8,
           "e4m3b15": torch.uint8}


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=CASES)
    ap.add_argument("nranks", type=int)
    ap.add_argument("bytes_per_rank", type=int)
    ap.add_argument("dtype", choices=sorted(STORAGE))
    ap.add_argument("--calls", type=int, default=3)
    a = ap.parse_args()
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    esize = torch.empty(0, dtype=STORAGE[a.dtype]).element_size()
    count = a.bytes_per_rank // esize
    g = torch.Generator(device=dev).manual_seed(0)
    if STORAGE[a.dtype] == torch.uint8:      # FP8 codes: small magnitudes, no NaN
        ins = [torch.randint(0, 0x60, (count,), dtype=torch.uint8, device=dev, generator=g) for _ in range(a.nranks)]
    else:
        ins = [torch.randn(count, dtype=STORAGE[a.dtype], device=dev, generator=g) for _ in range(a.nranks)]
    outs = [torch.empty_like(ins[0]) for _ in range(a.nranks)]
    want = [torch.empty_like(ins[0]) for _ in range(a.nranks)]
    nbp = sar.sar_ll_packet_bytes(count, a.dtype)
    pk = [torch.zeros(max(16, nbp), dtype=torch.uint8, device=dev) for _ in range(a.nranks)]
    res = torch.zeros(max(16, nbp), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    sar.sar_allreduce(ins, want, count=count, dtype=a.dtype)
    for epoch in range(1, a.calls + 1):
        if a.case in ("rsag", "rsag_two_phase", "ll_allpair"):
            algo = {"rsag": sar.SAR_ALGO_RSAG, "rsag_two_phase": sar.SAR_ALGO_RSAG_TWO_PHASE,
                    "ll_allpair": sar.SAR_ALGO_LL_ALLPAIR}[a.case]
            sar.sar_allreduce(ins, outs, count=count, dtype=a.dtype, algo=algo)
        elif a.case == "ll":
            sar.sar_allreduce_ll(ins, outs, pk, epoch, st, count=count, dtype=a.dtype)
        elif a.case == "ll_fused":
            sar.sar_allreduce_ll_fused(ins, outs, pk, st, epoch=epoch, count=count, dtype=a.dtype)
        elif a.case == "ll_cluster":
            sar.sar_allreduce_ll_cluster(ins, outs, st, count=count, dtype=a.dtype)
        else:
            sar.sar_allreduce_ll_writeback(ins, outs, pk, res, st, multi_dest=a.case.endswith("multi_dest"),
                                           epoch=epoch, count=count, dtype=a.dtype)
    torch.cuda.synchronize()
    if sar.sar_read_device_status(st) != sar.SAR_OK:
        raise SystemExit("profile_case: an LL poll timed out")
    if not all(torch.equal(o.view(torch.uint8), want[0].view(torch.uint8)) for o in outs):
        raise SystemExit("profile_case: outputs differ from the rsag allreduce")
    print(f"profile_case: {a.case} {a.nranks} x {a.bytes_per_rank} B {a.dtype}, {a.calls} calls OK")


if __name__ == "__main__":
    main()
