"""Plant plausible mistakes in copies of the oracle (on the CPU) and check the pins catch every one of them."""
import os
import subprocess
import sys

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "hs_oracle.c")

# (name, original text, replacement): each one a mistake a careful reader could make
MUTANTS = [
    ("tie_break_highest_slot", "return (x->slot > y->slot) - (x->slot < y->slot);",
     "return (x->slot < y->slot) - (x->slot > y->slot);"),
    ("most_recent_first", "if (x->stamp != y->stamp) return (x->stamp > y->stamp) - (x->stamp < y->stamp);",
     "if (x->stamp != y->stamp) return (x->stamp < y->stamp) - (x->stamp > y->stamp);"),
    ("misses_descending", "const int32_t t = miss[j], v = cand[j].slot",
     "const int32_t t = miss[m - 1 - j], v = cand[j].slot"),
    ("hit_not_restamped", "      slot_stamp[s] = step;\n      in_sel[s] = 1;", "      in_sel[s] = 1;"),
    ("fill_not_stamped", "    slot_stamp[v] = step;\n    if (hot)", "    if (hot)"),
    ("old_token_not_unmapped", "      tok2slot[u] = -1;\n", "\n"),
    ("selected_slots_evictable", "    if (!in_sel[v]) {", "    if (1) {"),
    ("wrong_host_row", "host_rows + (size_t)t * (size_t)row_bytes", "host_rows + (size_t)(t ^ 1) * (size_t)row_bytes"),
    ("duplicates_accepted", "err |= ORA_ERR_DUP;", ";"),
    ("hits_miscounted", "counters[0] += (uint64_t)hits;", "counters[0] += (uint64_t)m;"),
    ("evictions_miscounted", "      ++evictions;\n", "\n"),
    ("range_check_off_by_one", "if (sel[i] >= ctx) err |= ORA_ERR_RANGE;", "if (sel[i] > ctx) err |= ORA_ERR_RANGE;"),
    ("resident_fetched_anyway", "      ++inplace; /* served in place from the HBM-resident tier */",
     "      miss[m++] = t;"),
    ("resident_before_hot", "    if (s >= 0) {\n      slot_stamp[s] = step;\n      in_sel[s] = 1;\n      ++hits;\n    } else if",
     "    if (s >= 0 && !(resident && resident[t] >= 0)) {\n      slot_stamp[s] = step;\n      in_sel[s] = 1;\n      ++hits;\n    } else if"),
    ("resident_encoding_off_by_one", "out_slots[i] = -2 - resident[sel[i]];", "out_slots[i] = -1 - resident[sel[i]];"),
]


_CHILD = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, pins
lib = oracle.load_library({so!r})
caught = []
for pin in pins.ALL_PINS:
    try:
        pin(lib)
    except (AssertionError, IndexError, ValueError):
        caught.append(pin.__name__)
print("caught by:", caught)
sys.exit(1 if caught else 0)
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(mut), "-o", str(so)])
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _CHILD.format(root=os.path.dirname(tests_dir), tests=tests_dir, so=str(so))
    # a separate process: a planted mistake may also corrupt memory, which counts as caught
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin caught the planted mistake {name}: {r.stdout}{r.stderr}"
