"""Per-CTA timelines of back-to-back launches (observability tool).

Runs ``launches`` GEMMs back to back in one CUDA graph (programmatic dependent
launch edges kept, W rotated over copies larger than L2), each through
``lowm_gemm_bf16_debug(timeline=...)``, which records per CTA the
%globaltimer at the end of the prologue, the MMA warp's first and last full
stage and the end of the epilogue.  The analysis splits a steady-state GEMM
period into where its time goes:

    python -m split_bf16_gemm_swap_gb300.timeline --M 4 --N 6144 --K 4096 --split-k 2 --flags 1

Stamps are on the global timer, whose resolution is coarse (about 0.25 us on
GB300), so the output gives medians and spreads over many CTAs and GEMMs.
"""
from __future__ import annotations

import argparse
import json

import numpy as np

PROLOGUE, FIRST_FULL, LAST_FULL, EPILOGUE = range(4)


def analyse(T: np.ndarray, first: int = None, count: int = None) -> dict:
    """Phase statistics of a [launches, ctas, 4] array of timestamps in ns.

    Times of GEMM i are taken relative to the previous GEMM's last epilogue end
    ("prev_end"), the moment the whole previous launch has finished its work.
    """
    T = np.asarray(T, dtype=np.float64)
    G = T.shape[0]
    if first is None:
        first = G // 3
    if count is None:
        count = max(1, G - first - 1)
    rows = []
    for i in range(max(1, first), min(G, first + count)):
        a = T[i]
        ref = T[i - 1][:, EPILOGUE].max()
        rows.append({
            "prologue_end_med": np.median(a[:, PROLOGUE]) - ref,
            "first_full_med": np.median(a[:, FIRST_FULL]) - ref,
            "first_full_max": a[:, FIRST_FULL].max() - ref,
            "stream_med": np.median(a[:, LAST_FULL] - a[:, FIRST_FULL]),
            "last_full_to_epilogue_end_med": np.median(a[:, EPILOGUE] - a[:, LAST_FULL]),
            "epilogue_end_max": a[:, EPILOGUE].max() - ref,
            "placed_before_prev_end": int((a[:, PROLOGUE] < ref).sum()),
        })
    ends = np.array([T[i][:, EPILOGUE].max() for i in range(G)])
    periods = np.diff(ends)[max(0, first - 1):]
    out = {k: float(np.median([r[k] for r in rows])) / 1e3 for k in rows[0] if k != "placed_before_prev_end"}
    out["placed_before_prev_end"] = int(np.median([r["placed_before_prev_end"] for r in rows]))
    out["period_us"] = float(np.mean(periods)) / 1e3
    out["ctas"] = int(T.shape[1])
    return out


def capture(M: int, N: int, K: int, split_k: int, flags: int, launches: int, seed: int = 1234):
    """Run the graph of `launches` GEMMs twice and return the second replay's timestamps (ns)."""
    import torch
    from . import inputs, lowm
    st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, split_k, flags)
    if st != lowm.LOWM_OK:
        raise lowm.LowmError(st, "lowm_gemm_query_tactic_ex")
    ctas = t["ctas"]
    A, W = inputs.make_problem(M, N, K, seed=seed)
    Ad = A.cuda()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    R = max(2, -(-2 * l2 // (N * K * 2)) + 1)
    Ws = [W.cuda() for _ in range(R)]
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    tl = torch.zeros((launches, 4 * ctas), dtype=torch.int64, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        for i in range(launches):
            st = lowm.lowm_gemm_bf16_debug(Ad, Ws[i % R], C, M, N, K, split_k, s, timeline=tl[i], flags=flags)
            if st != lowm.LOWM_OK:
                raise lowm.LowmError(st, "lowm_gemm_bf16_debug")
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    st, detail = lowm.lowm_gemm_sync_status()
    if st != lowm.LOWM_OK:
        raise lowm.LowmError(st, "kernel status %#x" % detail)
    T = tl.cpu().numpy().reshape(launches, ctas, 4)
    return T, t


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--M", type=int, default=4)
    ap.add_argument("--N", type=int, default=6144)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--split-k", type=int, default=2)
    ap.add_argument("--flags", type=int, default=1, help="launch flags (1 = LOWM_FLAG_W_BEFORE_PDL_WAIT)")
    ap.add_argument("--launches", type=int, default=30)
    args = ap.parse_args(argv)
    from . import build
    build.build()
    T, tactic = capture(args.M, args.N, args.K, args.split_k, args.flags, args.launches)
    res = analyse(T)
    res["workload"] = "M%d N%d K%d split_k %d flags %d" % (args.M, args.N, args.K, tactic["split_k"], args.flags)
    res["ring"] = "%d x %d" % (tactic["kb_per_stage"], tactic["stages"])
    print(json.dumps({k: (round(v, 3) if isinstance(v, float) else v) for k, v in res.items()}))


if __name__ == "__main__":
    main()
