"""The oracle's expert FFNs evaluated in worker processes, for full-size
comparisons.

The main process draws each touched expert's fp32 weights with the same
generator the CUDA layer was built from (the GPU's), and a pool of spawned
workers (started before they could inherit a CUDA context) quantises them
with the oracle's own quantiser and returns swiglu_expert(rows, expert) in
fp64.  ``oracle.moe.forward`` then combines the results exactly as it does
with its own loop (its ``expert_fn`` hook)."""
import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np


def _expert_out(args):
    from oracle import moe
    from tests._oracle_layer import expert_from_fp32
    fmt, g, u, d, xr = args
    return moe.swiglu_expert(xr, expert_from_fp32(fmt, g, u, d))


class OraclePool:
    """Context manager: ``forward(x, ol, w)`` = oracle.moe.forward(x, ol) with
    the experts of workload ``w`` evaluated in parallel."""

    def __init__(self, workers=None):
        self.workers = workers or min(16, os.cpu_count() or 1)

    def __enter__(self):
        self.ex = cf.ProcessPoolExecutor(self.workers, mp_context=mp.get_context("spawn"))
        return self

    def __exit__(self, *a):
        self.ex.shutdown()

    def expert_outputs(self, x, r, w, device="cuda", chunk=32):
        """{e: z [M_e, H]} for the active experts of routing r."""
        from block_quantized_moe_layer_gb300 import synth
        x = np.asarray(x, np.float64)
        act = [int(e) for e in r["act"]]
        out = {}
        for i in range(0, len(act), chunk):
            tasks, es = [], act[i:i + chunk]
            for e in es:
                sl = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
                g, u, d = (t.float().cpu().numpy() for t in synth.expert(w, e, device))
                tasks.append((w.routed_fmt, g, u, d, x[sl // w.top_k]))
            for e, z in zip(es, self.ex.map(_expert_out, tasks)):
                out[e] = z
        return out

    def forward(self, x, ol, w, device="cuda", routing=None):
        from oracle import moe
        r = moe.route(np.asarray(x, np.float64), ol) if routing is None else routing
        zs = self.expert_outputs(x, r, w, device)
        return moe.forward(x, ol, routing=r, expert_fn=lambda e, xr: zs[e])

    def layer_forward(self, workload_of):
        """A ``layer_forward(x, ol)`` for oracle.mtp: ``workload_of`` maps id(ol)
        to the synth workload whose weights ol holds."""
        def fwd(x, ol):
            return self.forward(x, ol, workload_of[id(ol)])
        return fwd
