"""Writes the stored planted-token deltas of the peaked workloads (B=8 planted and the B=64 block-16
stress case) and their achieved statistics. Calls only the CPU oracle and the input generator.

The pages' Table 1 ("DFlash 2: keeping drafts parallel", section "正しいトークンはすでにそこに
あります") has the right token at the top with about 85 % of the mass and among the top 16 in about
99 % of slots. The workloads mimic that with a planted token per slot: its lm_head row W[p] is
moved by a delta D so that, at the slot's conv output row z_r (the row the LM head reads), its
logit becomes the log-sum-exp of the slot's other logits plus log(0.85 / 0.15) (85 % of the mass),
while its logits at every other row of the workload do not move:
    <z_m, D> = beta * [m == r] for all rows m,   beta = target - <z_r, W[p]>,
solved with the least norm, D = Z^T (Z Z^T)^-1 beta e_r, Z all the workload's conv output rows
(float64 from the oracle's bf16 output; an M x M system). The deltas are stored as 8-bit codes with a per-row step (the
planted rows are then bf16(W[p] + step * code)); the statistics below are measured on those final
rows, so the rounding of the codes and of the bf16 rows is part of what they report.

    python tests/golden/make_planted_rows.py
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import core as O  # noqa: E402

LEVELS = 127  # codes -127 .. 127


def solve_deltas(rc, inp, planted):
    sh = rc.shape
    z = O.conv_chain(inp["hidden"], inp["conv_w"], sh.dtype, sh.group_size)
    slots = np.argwhere(planted >= 0)  # row-major: the order synth applies them in
    ids = planted[planted >= 0]
    rows = np.stack([z[b, t] for b, t in slots])
    l32 = O.logits(rows, inp["lm_head"]).astype(np.float64)
    betas = np.zeros(len(ids))
    for i, p in enumerate(ids):
        l = l32[i]
        others = np.delete(l, p)
        m = others.max()
        lse_others = m + np.log(np.exp(others - m).sum())
        target = lse_others + np.log(synth.PLANT_MASS / (1.0 - synth.PLANT_MASS))
        betas[i] = target - l[p]
    T = sh.block
    Z = O.widen(z).reshape(-1, sh.hidden)  # [M, H], row m = b * T + t
    E = np.zeros((Z.shape[0], len(ids)))
    E[slots[:, 0] * T + slots[:, 1], np.arange(len(ids))] = betas
    deltas = (Z.T @ np.linalg.solve(Z @ Z.T, E)).T  # [n, H]
    return z, slots, ids, deltas, betas


def quantize(deltas):
    step = np.abs(deltas).max(axis=1) / LEVELS
    step[step == 0] = 1.0
    q = np.clip(np.rint(deltas / step[:, None]), -LEVELS, LEVELS).astype(np.int8)
    return q, step.astype(np.float64)


def statistics(rc, z, slots, ids, lm_head_planted, lm_head_drawn):
    """Achieved mass and top-16 membership of the planted token at its slot, and how far the
    planted rows moved the logits of the planted tokens at the other rows of their sequences."""
    rows = np.stack([z[b, t] for b, t in slots])
    l32 = O.logits(rows, lm_head_planted).astype(np.float64)
    mass, in_top, top1 = [], [], []
    for i, p in enumerate(ids):
        l = l32[i]
        m = l.max()
        lse = m + np.log(np.exp(l - m).sum())
        mass.append(float(np.exp(l[p] - lse)))
        order = np.argsort(-l, kind="stable")
        in_top.append(bool(p in order[:rc.shape.top_k]))
        top1.append(bool(order[0] == p))
    # leakage: each planted token's logit at every other row of the workload, before and after
    T = rc.shape.block
    zall = z.reshape(-1, rc.shape.hidden)
    before = O.logits(zall, lm_head_drawn[ids]).astype(np.float64)  # [M, n]
    after = O.logits(zall, lm_head_planted[ids]).astype(np.float64)
    own = slots[:, 0] * T + slots[:, 1]
    diff = np.abs(after - before)
    diff[own, np.arange(len(ids))] = 0.0
    moved = [float(diff.max())]
    return {"planted_slots": int(len(ids)), "slots": int(rc.shape.batch * T),
            "mass_mean": float(np.mean(mass)), "mass_min": float(np.min(mass)), "mass_max": float(np.max(mass)),
            "top1_frac": float(np.mean(top1)), "in_top16_frac": float(np.mean(in_top)),
            "other_rows_logit_moved_max": float(np.max(moved)),
            "other_rows_logit_moved_rms": float(np.sqrt(np.mean(diff ** 2)))}


def main():
    for config in (3, 5):
        rc = synth.recipe(config)
        inp = synth.make_inputs(rc, apply_planting=False)
        planted = synth.planted_slots(rc)
        z, slots, ids, deltas, betas = solve_deltas(rc, inp, planted)
        q, step = quantize(deltas)
        path = synth.planted_rows_path(rc)
        np.savez_compressed(path, ids=ids.astype(np.int32), q=q, step=step)
        drawn = inp["lm_head"].copy()
        synth.apply_planted_rows(rc, inp["lm_head"], planted)
        st = statistics(rc, z, slots, ids, inp["lm_head"], drawn)
        st["beta_mean"] = float(betas.mean())
        with open(path.replace(".npz", ".json"), "w") as f:
            json.dump(st, f, indent=1)
        print(rc.name, os.path.getsize(path), st, flush=True)


if __name__ == "__main__":
    main()
