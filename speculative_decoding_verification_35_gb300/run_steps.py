"""Run the verify step of one synthetic workload a few times through the C ABI (for profilers and checks).

    python -m speculative_decoding_verification_35_gb300.run_steps [WORKLOAD] [STEPS] [SHARDS]

One device copy of the workload's batch (seeded synthetic logits, see ``synth``), STEPS consecutive calls
of spec_verify_ex on the current stream, then one synchronisation; it fails if the device reports an
error. With SHARDS, the vocabulary-sharded step instead: the batch split into SHARDS contiguous vocabulary
slices held by this process, each step the four spec_shard_* calls per shard with the records stacked
between them. A profiler capture of one launch uses, e.g., ``-k regex:k_verify -s 2 -c 1`` over 3 steps.
"""
from __future__ import annotations

import sys

import numpy as np


def main(argv=None) -> int:
    import torch

    from . import specverify as sv
    from . import synth
    argv = sys.argv[1:] if argv is None else argv
    name = argv[0] if argv else synth.HEADLINE
    steps = int(argv[1]) if len(argv) > 1 else 3
    shards = int(argv[2]) if len(argv) > 2 else 0
    b = synth.make_batch(name)

    def logits(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()

    tgt, dft = logits(b.target), logits(b.draft)
    toks = torch.from_numpy(b.draft_tokens).cuda()
    offs = torch.from_numpy(b.seq_offsets).cuda()
    gam = torch.from_numpy(b.gammas).cuda()
    if shards:
        from .shard import CudaShard, local_steps
        bounds = [b.V * j // shards for j in range(shards + 1)]
        T = float(np.float32(b.temperature))
        sh = [CudaShard(j, bounds, tgt[:, bounds[j]:bounds[j + 1]].contiguous(),
                        None if dft is None or T == 0 else dft[:, bounds[j]:bounds[j + 1]].contiguous(),
                        toks, offs, gam, b.B, b.V, int(b.gammas.max()), b.R_t, b.R_d, T) for j in range(shards)]
        for i in range(steps):
            local_steps(sh, 1, i)
        torch.cuda.synchronize()
        bad = [int(x.status.item()) for x in sh if int(x.status.item())]
        if bad:
            raise RuntimeError(f"device status {bad[0]:#x}")
        print("ok", name, steps, "shards", shards)
        return 0
    call = sv.Call(b.B, b.V, int(b.gammas.max()), b.R_t, b.R_d)
    for i in range(steps):
        rc = call.run(tgt, dft, toks, offs, gam, b.temperature, 1, i, clear_status=False)
        if rc != sv.SV_OK:
            raise RuntimeError(sv.spec_verify_status_string(rc))
    torch.cuda.synchronize()
    if call.status_bits():
        raise RuntimeError(f"device status {call.status_bits():#x}")
    print("ok", name, steps)
    return 0


if __name__ == "__main__":
    sys.exit(main())
