"""Write tests/golden/segment_counts.json: the float64 oracle's number of
positive-length (ray, cell) pieces of every full-size workload, and of the
reduced parity cases.  Calls only the oracle and the input generators.

    python tests/golden/make_segment_counts.py [--threads N]
"""

import argparse
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import ctp_inputs as ci  # noqa: E402
import oracle  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--threads", type=int, default=0)
    ap.add_argument("--out", default=os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                  "segment_counts.json"))
    args = ap.parse_args()
    out = {"about": "Positive-length (ray, cell) pieces per pass, counted by the float64 "
                    "oracle (oracle.segment_count) on the seeded workloads of ctp_inputs.",
           "full": {}, "small": {}}
    for idx, w in ci.small_cases().items():
        scan = oracle.Scan.from_workload(w, ci.frames(w))
        out["small"][str(idx)] = {"name": w.name, "segments": oracle.segment_count(scan, threads=args.threads)}
    for idx, w in ci.WORKLOADS.items():
        t = time.time()
        scan = oracle.Scan.from_workload(w, ci.frames(w))
        n = oracle.segment_count(scan, threads=args.threads)
        out["full"][str(idx)] = {"name": w.name, "segments": n, "rays": w.n_rays}
        print(f"{w.name}: {n} segments in {time.time() - t:.1f} s", flush=True)
    with open(args.out, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")


if __name__ == "__main__":
    main()
