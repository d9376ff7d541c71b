"""Pins for the float64 oracle (CPU only).

The oracle restates the record / replay kernels of the "metaltile-std
gated_delta_replay.rs" page and the tiled repeat of the "mlx-native
repeat_tiled.rs" page.  Nothing here re-types the oracle's loops: each check
is something the pages or the mathematics fix independently --

* a worked example derived by hand (tests/golden/worked_example_dk2_dv2.json);
* closed forms: zero state with g = beta = 1 and unit k writes the outer
  product v (x) k and reads out v (k.q); g = 0 resets the row to beta v (x) k;
* the delta-rule projection identity after every step,
  s_new.k = g (1 - beta |k|^2) (s_old.k) + beta |k|^2 v;
* an independent matrix-form restatement of the step,
  S <- g S (I - beta k k^T) + beta v k^T, y = S q;
* replay invariants (accepted = T, accepted = a, accepted = 0, all masked,
  NaN in unused tape slots);
* equivariance under batch / value-row permutations, the block GQA mapping,
  and the tiled mapping as the pinned repeat followed by a record;
* per-sequence accepted counts against a record over each sequence's prefix;
* numpy fancy indexing for the repeat.

``test_pins_catch_planted_mistakes`` compiles mutated copies of the oracle
source (a dropped decay, a flipped sign, a wrong GQA index, ...) and checks
that every mutant fails at least one pin.
"""
from __future__ import annotations

import json
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_dk2_dv2.json")


# --------------------------------------------------------------- helpers
def _rand_case(seed, B=2, T=5, Hk=2, Hv=4, Dk=6, Dv=5, mask=None, unit_k=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hk, Dk))
    k = rng.standard_normal((B, T, Hk, Dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, Dv))
    g = rng.uniform(0.5, 1.0, (B, T, Hv))
    beta = rng.uniform(0.1, 1.0, (B, T, Hv))
    s = rng.standard_normal((B, Hv, Dv, Dk)) * 0.3
    m = None
    if mask == "random":
        m = (rng.random((B, T)) < 0.6).astype(np.uint32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, state=s, mask=m)


def _matrix_form(q, k, v, g, beta, state, mask):
    """Independent restatement: per (b, hv) the Dv x Dk matrix update
    S <- g S (I - beta k k^T) + beta v k^T, delta = beta (v - g S k), y = S q."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    grp = Hv // Hk
    S = state.copy()
    y = np.full((B, T, Hv, Dv), np.nan)
    dl = np.full((B, T, Hv, Dv), np.nan)
    eye = np.eye(Dk)
    for b in range(B):
        for hv in range(Hv):
            hk = hv // grp
            M = S[b, hv]
            for t in range(T):
                if mask is not None and mask[b, t] == 0:
                    continue
                kt, qt = k[b, t, hk], q[b, t, hk]
                gt, bt = g[b, t, hv], beta[b, t, hv]
                dl[b, t, hv] = bt * (v[b, t, hv] - gt * (M @ kt))
                M = gt * M @ (eye - bt * np.outer(kt, kt)) + bt * np.outer(v[b, t, hv], kt)
                y[b, t, hv] = M @ qt
            S[b, hv] = M
    return dict(y=y, delta_log=dl, state_out=S)


# ------------------------------------------------ individual pin checks
# Each check takes an oracle-like object (``record``/``replay``/``repeat_tiled``)
# so the same checks run against planted-mistake mutants below.

def check_worked_example(orc):
    gold = json.load(open(GOLDEN))
    inp = {kk: np.array(vv, dtype=np.float64) for kk, vv in gold["inputs"].items()}
    out = orc.record(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"])
    for name, want in gold["record"].items():
        np.testing.assert_array_equal(out[name], np.array(want), err_msg=name)
    gm = gold["record_masked"]
    mask = np.array(gm["mask"], dtype=np.uint32)
    out_m = orc.record(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state"], mask)
    np.testing.assert_array_equal(out_m["y"][0, 1, 0], gm["y_t1"])
    np.testing.assert_array_equal(out_m["delta_log"][0, 1, 0], gm["delta_log_t1"])
    np.testing.assert_array_equal(out_m["state_out"], np.array(gm["state_out"]))
    assert np.isnan(out_m["y"][0, 0]).all() and np.isnan(out_m["delta_log"][0, 0]).all()
    for acc in (0, 1, 2):
        st = orc.replay(out["delta_log"], out["k_log"], out["g_log"], inp["state"], accepted=acc)
        np.testing.assert_array_equal(st, np.array(gold["replay"][f"accepted_{acc}"]))


def check_closed_form_outer_product(orc):
    # s = 0, g = beta = 1, |k| = 1, T = 1: row dv becomes v[dv] * k and y = v (k.q)
    c = _rand_case(11, B=2, T=1, Hk=2, Hv=4, Dk=7, Dv=3, unit_k=True)
    c["g"][:] = 1.0
    c["beta"][:] = 1.0
    c["state"][:] = 0.0
    out = orc.record(**c)
    for b in range(2):
        for hv in range(4):
            kk, qq, vv = c["k"][b, 0, hv // 2], c["q"][b, 0, hv // 2], c["v"][b, 0, hv]
            np.testing.assert_allclose(out["state_out"][b, hv], np.outer(vv, kk), atol=1e-14)
            np.testing.assert_allclose(out["y"][b, 0, hv], vv * (kk @ qq), atol=1e-14)
            np.testing.assert_allclose(out["delta_log"][b, 0, hv], vv, atol=1e-14)


def check_reset(orc):
    # g = 0 wipes the old row: s_new = beta v (x) k, delta = beta v, y = s_new q
    c = _rand_case(12, B=1, T=1, Hk=1, Hv=2, Dk=5, Dv=4)
    c["g"][:] = 0.0
    out = orc.record(**c)
    for hv in range(2):
        kk, qq, vv, bt = c["k"][0, 0, 0], c["q"][0, 0, 0], c["v"][0, 0, hv], c["beta"][0, 0, hv]
        np.testing.assert_allclose(out["state_out"][0, hv], bt * np.outer(vv, kk), atol=1e-13)
        np.testing.assert_allclose(out["delta_log"][0, 0, hv], bt * vv, atol=1e-13)
        np.testing.assert_allclose(out["y"][0, 0, hv], bt * vv * (kk @ qq), atol=1e-13)


def check_projection_identity(orc):
    # chained single steps: after every step s_new.k = g(1-b|k|^2)(s_old.k) + b|k|^2 v
    c = _rand_case(13, B=2, T=6, Hk=1, Hv=2, Dk=8, Dv=3)
    s = c["state"]
    for t in range(6):
        sl = {kk: (vv[:, t:t + 1] if kk not in ("state", "mask") else vv) for kk, vv in c.items()}
        sl["state"] = s
        sl["mask"] = None
        out = orc.record(**sl)
        for b in range(2):
            for hv in range(2):
                kk = c["k"][b, t, 0]
                gt, bt = c["g"][b, t, hv], c["beta"][b, t, hv]
                n2 = kk @ kk
                lhs = out["state_out"][b, hv] @ kk
                rhs = gt * (1 - bt * n2) * (s[b, hv] @ kk) + bt * n2 * c["v"][b, t, hv]
                np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
        s = out["state_out"]
    # composition of single steps == one multi-step call
    full = orc.record(**c)
    np.testing.assert_allclose(full["state_out"], s, rtol=1e-12, atol=1e-12)


def check_matrix_form(orc):
    for seed, shp, mask in [(21, dict(B=1, T=3, Hk=1, Hv=1, Dk=4, Dv=4), None),
                            (22, dict(B=2, T=5, Hk=2, Hv=4, Dk=6, Dv=3), None),
                            (23, dict(B=3, T=7, Hk=1, Hv=3, Dk=5, Dv=8), "random"),
                            (24, dict(B=2, T=4, Hk=4, Hv=8, Dk=3, Dv=2), "random")]:
        c = _rand_case(seed, mask=mask, **shp)
        out = orc.record(**c)
        ref = _matrix_form(**c)
        for name in ("y", "delta_log", "state_out"):
            np.testing.assert_allclose(out[name], ref[name], rtol=1e-12, atol=1e-12,
                                       err_msg=f"{name} seed {seed}")


def check_replay_invariants(orc):
    c = _rand_case(31, B=3, T=6, Hk=1, Hv=2, Dk=5, Dv=4, mask="random")
    rec = orc.record(**c)
    tape = (rec["delta_log"], rec["k_log"], rec["g_log"])
    # accepted = T (and beyond) reproduces record
    for acc in (6, 9):
        st = orc.replay(*tape, c["state"], c["mask"], accepted=acc)
        np.testing.assert_allclose(st, rec["state_out"], rtol=1e-12, atol=1e-12)
    # accepted = a reproduces a record over the first a tokens
    for a in (1, 2, 4):
        sub = {kk: (vv[:, :a] if kk not in ("state",) and vv is not None else vv)
               for kk, vv in c.items()}
        rec_a = orc.record(**sub)
        st = orc.replay(*tape, c["state"], c["mask"], accepted=a)
        np.testing.assert_allclose(st, rec_a["state_out"], rtol=1e-12, atol=1e-12)
    # accepted = 0 and an all-off mask are the identity, bit for bit
    np.testing.assert_array_equal(orc.replay(*tape, c["state"], c["mask"], accepted=0), c["state"])
    off = np.zeros_like(c["mask"])
    np.testing.assert_array_equal(orc.replay(*tape, c["state"], off, accepted=6), c["state"])
    # masked / unaccepted tape slots may hold anything: the select never reads them
    assert np.isnan(rec["delta_log"][c["mask"] == 0]).all()
    st3 = orc.replay(*tape, c["state"], c["mask"], accepted=3)
    assert np.isfinite(st3).all()


def check_masked_steps(orc):
    c = _rand_case(41, B=2, T=4, Hk=1, Hv=2, Dk=4, Dv=3)
    c["mask"] = np.zeros((2, 4), dtype=np.uint32)
    out = orc.record(**c)
    np.testing.assert_array_equal(out["state_out"], c["state"])
    assert np.isnan(out["y"]).all() and np.isnan(out["delta_log"]).all()
    assert np.isnan(out["k_log"]).all() and np.isnan(out["g_log"]).all()
    # any nonzero mask value means "on"
    c["mask"][:] = 7
    on = orc.record(**c)
    c["mask"] = None
    ref = orc.record(**c)
    np.testing.assert_array_equal(on["state_out"], ref["state_out"])


def check_tape_capture(orc):
    c = _rand_case(51, B=2, T=3, Hk=2, Hv=6, Dk=4, Dv=2, mask="random")
    out = orc.record(**c)
    for b in range(2):
        for t in range(3):
            for hv in range(6):
                if c["mask"][b, t]:
                    np.testing.assert_array_equal(out["k_log"][b, t, hv], c["k"][b, t, hv // 3])
                    assert out["g_log"][b, t, hv] == c["g"][b, t, hv]
                else:
                    assert np.isnan(out["k_log"][b, t, hv]).all()


def check_gqa_block_mapping(orc):
    # head hv of a grouped run equals a single-head run on k/q head hv // (Hv/Hk)
    c = _rand_case(61, B=1, T=4, Hk=2, Hv=6, Dk=5, Dv=3)
    out = orc.record(**c)
    for hv in range(6):
        hk = hv // 3
        one = orc.record(c["q"][:, :, hk:hk + 1], c["k"][:, :, hk:hk + 1], c["v"][:, :, hv:hv + 1],
                         c["g"][:, :, hv:hv + 1], c["beta"][:, :, hv:hv + 1],
                         c["state"][:, hv:hv + 1])
        np.testing.assert_array_equal(out["state_out"][:, hv], one["state_out"][:, 0])
        np.testing.assert_array_equal(out["y"][:, :, hv], one["y"][:, :, 0])


def check_gqa_tiled_mapping(orc):
    # the tiled mapping is the tiled repeat (pinned by numpy indexing in
    # check_repeat) followed by a record on the expanded heads (Hk' = Hv)
    c = _rand_case(62, B=2, T=4, Hk=2, Hv=6, Dk=5, Dv=3, mask="random")
    out = orc.record(**c, gqa="tiled")
    B, T, Hk, Dk = c["q"].shape
    Hv = c["v"].shape[2]

    def expand(x):
        return orc.repeat_tiled(x.reshape(B * T, Hk, Dk), Hv).reshape(B, T, Hv, Dk)

    ref = orc.record(expand(c["q"]), expand(c["k"]), c["v"], c["g"], c["beta"], c["state"],
                     c["mask"])
    for name in ("y", "delta_log", "state_out", "k_log", "g_log"):
        np.testing.assert_array_equal(out[name], ref[name], err_msg=name)
    # and it differs from the block mapping on the same inputs
    blk = orc.record(**c)
    assert not np.allclose(blk["state_out"], out["state_out"])


def check_replay_per_sequence(orc):
    # sequence b with its own accepted count a_b ends where a record over its
    # first a_b tokens ends; negative counts accept nothing, counts past T
    # accept everything
    c = _rand_case(33, B=5, T=6, Hk=1, Hv=2, Dk=4, Dv=3, mask="random")
    rec = orc.record(**c)
    tape = (rec["delta_log"], rec["k_log"], rec["g_log"])
    acc = np.array([0, 6, 3, -2, 9])
    st = orc.replay(*tape, c["state"], c["mask"], accepted=acc)
    for b in range(5):
        a = int(min(max(acc[b], 0), 6))
        if a == 0:
            np.testing.assert_array_equal(st[b], c["state"][b])
            continue
        sub = {kk: (vv[b:b + 1] if kk == "state" else vv[b:b + 1, :a]) if vv is not None else None
               for kk, vv in c.items()}
        np.testing.assert_allclose(st[b], orc.record(**sub)["state_out"][0],
                                   rtol=1e-12, atol=1e-12, err_msg=f"sequence {b}")


def check_permutation_equivariance(orc):
    c = _rand_case(71, B=3, T=4, Hk=1, Hv=2, Dk=5, Dv=6, mask="random")
    out = orc.record(**c)
    pb = np.array([2, 0, 1])
    cb = {kk: (vv[pb] if vv is not None else None) for kk, vv in c.items()}
    ob = orc.record(**cb)
    for name in ("y", "delta_log", "state_out"):
        np.testing.assert_array_equal(ob[name], out[name][pb])
    pr = np.array([3, 5, 0, 1, 4, 2])          # permute value rows dv
    cr = dict(c)
    cr["v"] = c["v"][..., pr]
    cr["state"] = c["state"][:, :, pr]
    orr = orc.record(**cr)
    np.testing.assert_array_equal(orr["state_out"], out["state_out"][:, :, pr])
    np.testing.assert_array_equal(orr["y"], out["y"][..., pr])


def check_repeat(orc):
    rng = np.random.default_rng(81)
    for seq, hg, h, kd, dt in [(5, 2, 6, 4, np.float32), (3, 4, 4, 8, np.uint16),
                               (2, 1, 5, 3, np.float16), (7, 3, 12, 1, np.float64)]:
        src = (rng.standard_normal((seq, hg, kd)) * 100).astype(dt)
        np.testing.assert_array_equal(orc.repeat_tiled(src, h), src[:, np.arange(h) % hg, :])


ALL_CHECKS = [check_worked_example, check_closed_form_outer_product, check_reset,
              check_projection_identity, check_matrix_form, check_replay_invariants,
              check_masked_steps, check_tape_capture, check_gqa_block_mapping,
              check_gqa_tiled_mapping, check_replay_per_sequence,
              check_permutation_equivariance, check_repeat]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle.default())


# -------------------------------------------------- planted-mistake mutants
MUTANTS = {
    "drop_decay": ("s[i] = s[i] * gt;", "s[i] = s[i];"),
    "delta_sign": ("const double delta = (v[vi] - kv) * bt;", "const double delta = (kv - v[vi]) * bt;"),
    "readout_before_update": ("s[i] = s[i] + kt[i] * delta;\n                    out += s[i] * qt[i];",
                              "out += s[i] * qt[i];\n                    s[i] = s[i] + kt[i] * delta;"),
    "tiled_instead_of_block_gqa": ("tiled_gqa ? hv % Hk : hv / group;", "hv % Hk;"),
    "block_instead_of_tiled_gqa": ("tiled_gqa ? hv % Hk : hv / group;", "hv / group;"),
    "per_seq_accepted_of_first_sequence": ("accepted_per_seq ? accepted_per_seq[b] : accepted;",
                                           "accepted_per_seq ? accepted_per_seq[0] : accepted;"),
    "beta_dropped": ("const double delta = (v[vi] - kv) * bt;", "const double delta = (v[vi] - kv);"),
    "q_for_k_in_kv": ("kv += s[i] * kt[i];", "kv += s[i] * qt[i];"),
    "state_transposed": ("const double *row_in = state_in + (n * Dv + dv) * Dk;\n            for (int64_t i = 0; i < Dk; ++i) s[i] = row_in[i];\n            for (int64_t t = 0; t < T; ++t) {\n                const uint32_t m = mask ? mask[b * T + t] : 1u;\n                if (m == 0) continue;",
                         "const double *row_in = state_in + n * Dv * Dk;\n            for (int64_t i = 0; i < Dk; ++i) s[i] = row_in[i * Dv + dv];\n            for (int64_t t = 0; t < T; ++t) {\n                const uint32_t m = mask ? mask[b * T + t] : 1u;\n                if (m == 0) continue;"),
    "record_ignores_mask": ("                if (m == 0) continue;\n                const double *kt", "                (void)m;\n                const double *kt"),
    "replay_ignores_accepted": ("const int do_step = (t < acc) && (m != 0);", "const int do_step = (m != 0);"),
    "replay_ignores_mask": ("const int do_step = (t < acc) && (m != 0);", "const int do_step = (t < acc);"),
    "replay_additive_decay": ("s[i] = s[i] * gt + kt[i] * d;", "s[i] = s[i] + gt * kt[i] * d;"),
    "repeat_block_mapping": ("(t * hg + hh % hg) * kdim", "(t * hg + hh / (h / hg)) * kdim"),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(mutant, tmp_path):
    old, new = MUTANTS[mutant]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {mutant} not found exactly once"
    path = tmp_path / f"mut_{mutant}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.OracleLib(oracle.compile_c(str(path), str(tmp_path / f"lib_{mutant}.so")))
    caught = []
    for check in ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(lib)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin fails for planted mistake {mutant}"


def test_input_recipe_is_reproducible():
    a = workloads.make_config("tiny_f32")
    b = workloads.make_config("tiny_f32")
    for name in ("q", "k", "v", "g", "beta", "state"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name))
    # q/k rows are unit-norm in float32 before the cast
    n = np.linalg.norm(a.k.astype(np.float64), axis=-1)
    np.testing.assert_allclose(n, 1.0, rtol=1e-6)
    c = workloads.make_config("spec_verify_b16_t8_bf16", batch=2)
    assert c.k.dtype == np.uint16 and 0 <= c.accepted <= 8
    lens = c.mask.sum(axis=1)
    assert ((lens >= 1) & (lens <= 8)).all()


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 1e-30, 3.0e38], dtype=np.float32)
    bits = workloads.f32_to_bf16_bits(x)
    back = workloads.bf16_bits_to_f32(bits)
    # halfway cases go to the even neighbour; exact values survive
    np.testing.assert_array_equal(back[:4], np.array([1.0, 1.0, 1.0 + 2 * 2.0 ** -7, -2.5], np.float32))
    assert abs(back[4] - 1e-30) / 1e-30 < 2.0 ** -8
