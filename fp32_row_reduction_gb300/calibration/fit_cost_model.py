"""Fit the plan cost model's constants to measured plan sweeps, then score the
frozen model on held-out shapes ("Whole-launch reduction cost policy": a fit
on calibration shapes only, leave the benchmark shapes out, report the
regret of the model's choice; "TIRx Metal reduction lowering" §6: the model
ranks legal candidates, measurement never selects a call's plan).

    python -m fp32_row_reduction_gb300.calibration.fit_cost_model \\
        --cal sweep_cal.jsonl.gz --held sweep_held.jsonl.gz

The model itself is the library's (tr_plan_estimate_with): this script only
searches its constants. Regret of a case = time of the plan with the lowest
estimate / time of the fastest measured plan - 1. The fit minimises the mean
regret over the calibration cases by coordinate descent on multiplicative
steps; the clock stays at its datasheet value and the segments plans' per-row
step (fitted on its own comparison with the split plans) is left as it is.
"""
import argparse
import collections
import gzip
import json
import math

import fp32_row_reduction_gb300 as tr

NAMES = ["launch", "latency", "cta_barrier", "cluster_barrier", "l2_over_hbm", "staged_row", "one_wave_alu", "wave",
         "slot_pass", "param_trip", "clock_ghz", "split_sync", "pair_overlap", "wave_slot_pass", "wave_row_share",
         "seg_row"]
# the clock is the datasheet value; the segments plans' per-row step is fitted on
# its own comparison with the split plans (the sweeps hold no segments plans)
FIXED = {"clock_ghz", "seg_row"}
PLAN_KEYS = ["op", "order", "kind", "lanes_per_row", "warps_per_row", "rows_per_cta", "cluster_ctas", "vec_slots",
             "block_threads", "ctas_per_sm", "grid_ctas", "flags", "resident_ctas"]


def load(path):
    """Sweep records, keeping the plans the library's current legality rules
    accept (occupancy aside: the sweep recorded the device's own)."""
    cases = collections.defaultdict(list)
    dev = tr.gb300_device_desc()
    opener = gzip.open if path.endswith(".gz") else open
    with opener(path, "rt") as f:
        for line in f:
            r = json.loads(line)
            p = tr.tr_plan(**{k: r["plan"][k] for k in PLAN_KEYS})
            q = tr.tr_plan(**{k: r["plan"][k] for k in PLAN_KEYS})
            st, why = tr.check_plan_for(dev, q, r["rows"], r["cols"], 1)
            if st != tr.TR_OK and "resident" not in why:
                continue
            cases[(r["op"], r["rows"], r["cols"])].append((r["us"], p))
    return cases


def pick_key(dev, plan, rows, cols, consts):
    """The library's ranking: the estimate (to 0.01 us), then its tie-break."""
    est = tr.estimate_with(dev, plan, rows, cols, 1, consts)
    warps = min(64, plan.resident_ctas * (plan.block_threads // 32) // max(1, dev.sm_count))
    return (round(est * 100.0), -warps, plan.warps_per_row * plan.cluster_ctas, plan.block_threads, plan.vec_slots)


def regrets(cases, consts, dev):
    out = {}
    for key, runs in cases.items():
        _, rows, cols = key
        best = min(us for us, _ in runs)
        pick = min(runs, key=lambda up: pick_key(dev, up[1], rows, cols, consts))
        out[key] = pick[0] / best - 1.0
    return out


def objective(cases, consts, dev):
    r = regrets(cases, consts, dev)
    return sum(r.values()) / len(r)


def fit(cases, start, dev, rounds=8):
    c = list(start)
    cur = objective(cases, c, dev)
    for _ in range(rounds):
        improved = False
        for i, name in enumerate(NAMES):
            if name in FIXED:
                continue
            for step in (4.0, 2.0, 1.5, 1.2, 1.1, 1.05):
                for f in (step, 1.0 / step):
                    trial = list(c)
                    trial[i] = c[i] * f if c[i] > 0 else 0.01
                    v = objective(cases, trial, dev)
                    if v < cur - 1e-9:
                        c, cur, improved = trial, v, True
        if not improved:
            break
    return c, cur


def report(name, cases, consts, dev):
    r = regrets(cases, consts, dev)
    vals = sorted(r.values())
    print(f"{name}: {len(vals)} cases, mean regret {100 * sum(vals) / len(vals):.1f}%, "
          f"max {100 * vals[-1]:.1f}%")
    for key in sorted(r, key=lambda k: -r[k])[:8]:
        print(f"   {key}: {100 * r[key]:.1f}%")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--cal", required=True)
    ap.add_argument("--held", required=True)
    args = ap.parse_args()
    tr.load()
    dev = tr.gb300_device_desc()
    cal, held = load(args.cal), load(args.held)
    start = tr.cost_constants()
    report("calibration, library constants", cal, start, dev)
    report("held out, library constants", held, start, dev)
    consts, _ = fit(cal, start, dev)
    print("fitted constants:")
    for n, v in zip(NAMES, consts):
        print(f"   {n} = {v!r}")
    report("calibration, fitted", cal, consts, dev)
    report("held out, fitted (frozen before scoring)", held, consts, dev)


if __name__ == "__main__":
    main()
