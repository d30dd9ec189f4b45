"""Each plausible slip planted in a copy of the oracle must fail a pin.

The mutants are text edits of ``oracle/a2a_oracle.c`` confined to one
function; each is compiled on the CPU into a temporary library and the pins
run against it in a child process (a mutant may crash), which must fail.
"""
import os
import re
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))

# (function, original text, planted slip, what kind of slip)
MUTANTS = [
    ("oracle_combine", "(d * S + s)) * H", "(s * W + d)) * H", "wrong source row"),
    ("oracle_combine", "(r * H + h)) * D", "(h * W + r)) * D", "transposed column group"),
    ("oracle_combine", "(r * (S * W) + (d * S + s))", "(r * (S * W) + (d * S))",
     "dropped row term"),
    ("oracle_combine", "(d * S + s) * (H * W)", "(d * S + s) * (H)", "wrong output row stride"),
    ("oracle_dispatch", "(r * S + (d * Sp + sp))", "(r * S + (sp * W + d))", "wrong source row"),
    ("oracle_dispatch", "(r * H + h)) * D", "(d * H + h)) * D", "wrong column group"),
    ("oracle_combine_back", "(r * H + h)) * D", "(d * H + h)) * D", "wrong column group"),
    ("oracle_combine_back", "(d * Sp + sp)) * H", "(sp * W + d)) * H", "wrong output row"),
    ("oracle_pc_replay", "(rank * H + h) * D + x;\n                        memcpy(peer",
     "(target * H + h) * D + x;\n                        memcpy(peer", "staging column"),
    ("oracle_pc_replay", "(buf * tasks + rank * nbd * H + hd) * 8;",
     "(buf * tasks + target * nbd * H + hd) * 8;", "producer wait slot index"),
    ("oracle_pc_replay", "(buf * tasks + r * nbd * H + hd) * 8] = 0;",
     "(buf * tasks + r * nbd * H) * 8] = 0;", "consumer reset slot index"),
    ("oracle_pc_replay", "const int64_t i_c = ((rank * S + s)", "const int64_t i_c = ((r * S + s)",
     "consumer output rank"),
    ("oracle_heap_at", "pe * slab_stride + offset", "pe * slab_stride", "dropped offset"),
    ("oracle_signal_op", "(uint64_t)cur + (uint64_t)value", "(uint64_t)value", "ADD acts as SET"),
    ("oracle_wait_satisfied", "current > value", "current >= value", "GT as GE"),
    ("oracle_wait_satisfied", "current < value", "current > value", "LT as GT"),
    ("oracle_alltoallv", "first += counts[r * W + e];", "first += counts[e * W + d];",
     "transposed send offset"),
    ("oracle_alltoallv", "(d * out_rows + pos) * row_bytes", "(d * out_rows + i) * row_bytes",
     "receive offset dropped"),
    ("oracle_alltoallv", "for (int64_t e = 0; e < d; e++)", "for (int64_t e = 0; e <= d; e++)",
     "off-by-one send offset"),
    ("oracle_allgather", "(d * W + r) * bytes", "(r * W + d) * bytes", "transposed gather"),
    ("oracle_two_phase_replay", "(rank * S + s0) * row;", "(target * S + s0) * row;",
     "bulk slot of the receiver"),
    ("oracle_two_phase_replay", "first_row = buf * block_s;", "first_row = s0;",
     "self buffer read as bulk"),
    ("oracle_two_phase_replay", "(buf * block_s + i) * row + h * D + x;",
     "(s0 + i) * row + h * D + x;", "self buffer written as bulk"),
    ("oracle_two_phase_replay", "(bs * W + rank) * 8;", "(bs * W + target) * 8;",
     "region-A slot of the receiver"),
    ("oracle_two_phase_replay", "if (r == rank) *slot = 0;", ";", "no credit return"),
    ("oracle_ag_matmul", "gather[(d * m_total + r * m_local + i) * k + x]",
     "gather[(d * m_total + d * m_local + i) * k + x]", "gather row of the receiver"),
    ("oracle_ag_matmul", "b[(d * k + x) * n + j]", "b[(d * k + j) * n + x]", "transposed b"),
    ("oracle_ag_matmul", "for (int64_t x = 0; x < k; x++)\n                    acc",
     "for (int64_t x = 1; x < k; x++)\n                    acc", "dropped first k term"),
    ("oracle_ag_matmul_at", "a[(r * m_local + row) * k + x]", "a[(d * m_local + row) * k + x]",
     "sampled row from the receiver"),
]


def _function_span(src: str, name: str):
    m = re.search(r"^[a-z].*\b" + name + r"\(", src, re.M)
    assert m, name
    start = m.start()
    nxt = re.search(r"^}\s*$", src[start:], re.M)
    return start, start + nxt.end()


def _mutate(src: str, func: str, old: str, new: str) -> str:
    a, b = _function_span(src, func)
    body = src[a:b]
    assert old in body, (func, old)
    return src[:a] + body.replace(old, new, 1) + src[b:]


@pytest.mark.parametrize("func,old,new,kind", MUTANTS, ids=[m[3] + "@" + m[0] for m in MUTANTS])
def test_mutant_is_caught(func, old, new, kind, tmp_path):
    with open(oracle.oracle.SOURCE) as f:
        src = f.read()
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(_mutate(src, func, old, new))
    lib = oracle.build(str(mutant_c), str(tmp_path / "libmutant.so"), force=True, werror=False)
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import oracle, oracle_pins\n"
        "oracle_pins.run_all(oracle.load(%r))\n" % (ROOT, HERE, lib)
    )
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert res.returncode != 0, f"planted slip '{kind}' in {func} passed every pin"


def test_unmutated_copy_passes(tmp_path):
    """Control: the same harness on an unchanged copy passes."""
    lib = oracle.build(oracle.oracle.SOURCE, str(tmp_path / "libcopy.so"), force=True)
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import oracle, oracle_pins\n"
        "oracle_pins.run_all(oracle.load(%r))\n" % (ROOT, HERE, lib)
    )
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
