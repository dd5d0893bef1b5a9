"""The pins must catch plausible mistakes planted in copies of the oracle (CPU only).

Each mutant is a copy of an oracle routine with one mistake (dropped term, wrong sign or
index, swapped operand). The pin checks of ``test_oracle_attention`` are run against it and
at least one must fail. The oracle itself is never modified.
"""
import math
import os
import subprocess

import numpy as np
import pytest

from oracle import attention as att
from oracle import native
from tests.test_oracle_attention import make_problem, sdpa


def pin_checks(fn):
    """Run the core pins against a decode implementation; return the names of those that fail."""
    failed = []
    P = make_problem(7, [1, 17, 100, 53, 250], 8, 2, 64, 16, "bf16")
    with np.errstate(all="ignore"):
        out = fn(P["q"], P["kc"], P["vc"], P["tables"], P["lens"], P["scale"])
        if not np.allclose(out, sdpa(P), rtol=0, atol=1e-12):
            failed.append("sdpa")
        P1 = make_problem(5, [1, 1], 8, 2, 64, 16, "bf16")
        o1 = fn(P1["q"], P1["kc"], P1["vc"], P1["tables"], P1["lens"], P1["scale"])
        if not all(np.array_equal(o1[b, j], att.to_f64(P1["logical"][b][1][0, j // 4]))
                   for b in range(2) for j in range(8)):
            failed.append("single_token")
        if getattr(fn, "supports_window", False):
            Pw = make_problem(17, [300, 40], 8, 2, 64, 16, "bf16")
            ow = fn(Pw["q"], Pw["kc"], Pw["vc"], Pw["tables"], Pw["lens"], Pw["scale"], window=50)
            sl = dict(Pw)
            sl["logical"] = [(k[-50:], v[-50:]) for k, v in Pw["logical"]]
            sl["lens"] = np.minimum(Pw["lens"], 50)
            if not np.allclose(ow, sdpa(sl), rtol=0, atol=1e-12):
                failed.append("window")
        Px = make_problem(13, [300, 7], 8, 2, 64, 16, "f32")
        Px["q"] = (Px["q"] * 100.0).astype(np.float32)
        ox = fn(Px["q"], Px["kc"], Px["vc"], Px["tables"], Px["lens"], Px["scale"])
        if not (np.isfinite(ox).all() and np.allclose(ox, sdpa(Px), rtol=0, atol=1e-11)):
            failed.append("extreme")
    return failed


# ---- NumPy mutants: each replaces one line of the definition ----------------------------------------

def _mutant(kind):
    def gather(cache, table, length, kv_head):
        B = cache.shape[2]
        if kind == "block_index":
            rows = [cache[int(table[min(t + 1, length - 1) // B]), kv_head, t % B, :] for t in range(length)]
        elif kind == "offset":
            rows = [cache[int(table[t // B]), kv_head, (B - 1 - t % B), :] for t in range(length)]
        elif kind == "drop_last":
            rows = [cache[int(table[t // B]), kv_head, t % B, :] for t in range(max(length - 1, 1))]
        else:
            rows = [cache[int(table[t // B]), kv_head, t % B, :] for t in range(length)]
        return att.to_f64(np.stack(rows))

    def dense(q, K, V, scale):
        s = (K @ q) if kind == "no_scale" else scale * (K @ q)
        m = 0.0 if kind == "no_max" else s.max()
        p = np.exp(s - m)
        if kind == "no_norm":
            return p @ V
        if kind == "swap_kv":
            s = scale * (V @ q)
            p = np.exp(s - s.max())
            return (p @ K) / p.sum()
        return (p @ V) / p.sum()

    def decode(q, k_cache, v_cache, tables, lens, scale):
        n, Hq, D = q.shape
        Hkv = k_cache.shape[1]
        g = Hq // Hkv
        qd = att.to_f64(q)
        out = np.zeros((n, Hq, D))
        for b in range(n):
            L = int(lens[b])
            for j in range(Hq):
                h = (j % Hkv) if kind == "gqa_mod" else j // g
                out[b, j] = dense(qd[b, j], gather(k_cache, tables[b], L, h), gather(v_cache, tables[b], L, h), scale)
        return out
    return decode


def _windowed(fn):
    fn.supports_window = True
    return fn


def test_unmodified_oracles_pass_every_pin():
    assert pin_checks(_windowed(lambda *a, **k: att.paged_decode(*a, **k))) == []
    assert pin_checks(_windowed(lambda *a, **k: native.decode(*a, **k))) == []


@pytest.mark.parametrize("kind", ["block_index", "offset", "drop_last", "no_scale", "no_max", "no_norm",
                                  "swap_kv", "gqa_mod"])
def test_numpy_mutant_is_caught(kind):
    assert pin_checks(_mutant(kind)) != []


# ---- C mutants: one textual edit of decode_ref.c, built into a temporary directory ------------------

C_MUTANTS = {
    "offset": ("(pos % block_size)) * D;", "(block_size - 1 - pos % block_size)) * D;"),
    "window_off_by_one": ("? len - window : 0;", "? len - window + 1 : 0;"),
    "gqa_mod": ("const int h = j / g;", "const int h = j % num_kv_heads;"),
    "no_scale": ("s[t] = scale * acc;", "s[t] = acc;"),
    "no_max": ("s[t] = exp(s[t] - m);", "s[t] = exp(s[t]);"),
    "no_norm": ("for (int d = 0; d < D; ++d) o[d] /= l;", ""),
    "swap_kv": ("K[(size_t)t * D + d] = load_value(k_cache", "K[(size_t)t * D + d] = load_value(v_cache"),
    "dtype_shift": ("<< 16;", "<< 15;"),
    "q_row": ("((size_t)b * num_q_heads + j) * D + d", "((size_t)b * num_q_heads + h) * D + d"),
}


@pytest.mark.parametrize("kind", sorted(C_MUTANTS))
def test_c_mutant_is_caught(kind, tmp_path):
    src = open(os.path.join(os.path.dirname(native.__file__), "decode_ref.c")).read()
    head, tail = src.split("int oracle_prefill", 1)      # mutate the decode routine only
    old, new = C_MUTANTS[kind]
    assert head.count(old) == 1, kind
    mpath = tmp_path / "mutant.c"
    mpath.write_text(head.replace(old, new) + "int oracle_prefill" + tail)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", str(so), str(mpath), "-lm"], check=True)
    assert pin_checks(_windowed(native.decode_fn_from(str(so)))) != []


# ---- allocator mutants: the batched decode-step append ----------------------------------------------

from oracle import alloc_model as am  # noqa: E402
from tests.test_oracle_alloc import append_pin_failures  # noqa: E402


def _append_mutant(kind):
    class Mutant(am.PoolModel):
        def append(self, seqs):
            seqs = [int(s) for s in seqs]
            if kind != "no_dup_check" and len(set(seqs)) != len(seqs):
                return am.ERR_INVALID, [], []
            if any(s not in self.tables for s in seqs):
                return am.ERR_NO_SEQ, [], []
            if any(-(-(self.lens[s] + 1) // self.B) > self.MB for s in seqs):
                return am.ERR_CAPACITY, [], []
            if self.fail_after >= 0 and self.n_allocs >= self.fail_after:
                return am.ERR_NO_BLOCKS, [], []
            rc = list(self.refcount)
            need = 0
            for s in seqs:
                if self.lens[s] % self.B == 0:
                    need += 0 if kind == "no_new_block" else 1
                elif rc[self.tables[s][-1]] > 1:
                    if kind != "no_replay":
                        rc[self.tables[s][-1]] -= 1
                    need += 1
            if kind != "no_precheck" and need > len(self.free):
                return am.ERR_NO_BLOCKS, [], []
            slots, pairs = [], []
            for s in seqs:
                st, _, sl, pr = self.alloc(s, 1)
                if st != am.OK:              # without the precheck a step can stop half-way
                    return st, slots, pairs
                if kind != "count_per_seq":
                    self.n_allocs -= 1
                slots += sl
                pairs += pr
            if kind != "count_per_seq":
                self.n_allocs += 1
            return am.OK, slots, pairs
    return Mutant


@pytest.mark.parametrize("kind", ["no_replay", "no_new_block", "no_precheck", "count_per_seq", "no_dup_check"])
def test_append_mutant_is_caught(kind):
    assert append_pin_failures(_append_mutant(kind)) != []


def test_append_mutant_copy_is_faithful():
    """The mutant template with no mistake planted passes every pin (so a caught mutant is caught
    for its planted mistake)."""
    assert append_pin_failures(_append_mutant("none")) == []
