"""Planted mistakes: each mutant is the oracle's own source with one plausible
error written in (a dropped term, a wrong sign, index or operand, a wrong
rounding rule). Every mutant must fail at least one pin, which shows that the
pins constrain each part of the oracle. Mutants run on the CPU only."""
import types

import pytest

from oracle import nvfp4_moe as O
from tests import oracle_pins as P
from tests.test_oracle import PINS

MUTATIONS = {
    "scale divisor 4 instead of 6": ("amax / np.float32(6.0)", "amax / np.float32(4.0)"),
    "e2m1 ties away from zero": ("np.rint(a / step)", "np.floor(a / step + 0.5)"),
    "e2m1 value table": ("2.0, 3.0, 4.0, 6.0]", "2.0, 3.0, 4.0, 5.0]"),
    "e4m3 truncates": ("r = np.rint(v / q) * q", "r = np.floor(v / q) * q"),
    "e4m3 bias off by one": ("np.exp2(e - 7.0)", "np.exp2(e - 8.0)"),
    "bf16 keeps an extra bit": ("q = np.exp2(e - 7.0)                    # spacing: 7",
                                "q = np.exp2(e - 8.0)                    # spacing: 7"),
    "atom slab strides swapped": ("(m % 32) * 16 + ((m // 32) % 4) * 4", "(m % 32) * 4 + ((m // 32) % 4) * 16"),
    "atoms along rows first": ("atom = (m // 128) * (Kc // 4) + c // 4", "atom = (c // 4) * 2 + m // 128"),
    "nibble order swapped": ("(c[..., 0::2] | (c[..., 1::2] << 4))", "(c[..., 1::2] | (c[..., 0::2] << 4))"),
    "weight rows reversed": ("D[r0:r1] = A[r0:r1] @ W.T", "D[r0:r1] = A[r0:r1] @ W[::-1].T"),
    "gate/up globals swapped": ("gate = d13[r0:r1, :I] * gg[e, 0]", "gate = d13[r0:r1, :I] * gg[e, 1]"),
    "up global dropped": ("up = d13[r0:r1, I:] * gg[e, 1]", "up = d13[r0:r1, I:]"),
    "silu sign error": ("gate / (1.0 + np.exp(-gate)) * up", "gate / (1.0 + np.exp(gate)) * up"),
    "down global dropped": ("y[t] += (w[slot] * gd[e]) * d2[r]", "y[t] += w[slot] * d2[r]"),
    "token index modulo": ("t, e = int(slot) // k", "t, e = int(slot) % T"),
    "rows visited backwards": ("for slot, e in enumerate(ids):", "for slot, e in reversed(list(enumerate(ids))):"),
    "groups in first-seen order": ("group_expert = sorted(rows_of)", "group_expert = list(rows_of)"),
    "gather by slot modulo": ("[np.asarray(row_slot) // k]", "[np.asarray(row_slot) % k]"),
    "GEMV path rounds its activations": ("A = bf16_bits_to_f64(np.asarray(a_bits, dtype=np.uint16))",
                                         "A = np.round(bf16_bits_to_f64(np.asarray(a_bits, dtype=np.uint16)) * 8) / 8"),
    "GEMV path reads K backwards": ("D[r0:r1] = A[r0:r1] @ Wg.T", "D[r0:r1] = A[r0:r1] @ Wg[:, ::-1].T"),
    "GEMV layer quantizes x": ("d13 = grouped_gemv_w4a16(xg, offs,", "d13 = grouped_gemv_w4a16(np.asarray(xg) & np.uint16(0xFFF0), offs,"),
    "zero block keeps codes": ("np.where((d == 0)[..., None], np.uint8(0), ", "np.where((d < 0)[..., None], np.uint8(0), "),
}


def make_mutant(old: str, new: str):
    with open(O.__file__) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation site not found: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(name, pages):
    M = make_mutant(*MUTATIONS[name])
    checks = [lambda m, p=p: p(m) for p in PINS] + [
        lambda m: P.check_e4m3_fold_figures(m, pages),
        lambda m: P.check_quantize_bytes(m, pages),
    ]
    for check in checks:
        try:
            check(M)
        except Exception:
            return
    pytest.fail(f"no pin caught the mutant: {name}")
