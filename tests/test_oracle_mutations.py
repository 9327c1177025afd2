"""Planted mistakes in the CPU oracle must each trip at least one pin.

Each case copies ``oracle/kv_oracle.c``, changes one expression to a plausible
mistake (a wrong index, a transposed operand, a dropped term, an off-by-one,
a swapped argument), compiles the copy into a temporary directory with gcc and
runs the pin battery against it in a child process (a planted mistake may write
out of bounds and crash; a crash counts as caught).  This shows the pins can tell a right oracle
from a wrong one; the real oracle passing them is ``test_oracle_pins.py``.
Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins

MUTATIONS = {
    "dev_hnd_index_swapped": ("inner = h * g->T + t;                /* [H][T] */",
                              "inner = t * g->T + h;                /* [H][T] */"),
    "dev_nhd_wrong_stride": ("inner = t * g->H + h;                /* [T][H] */",
                             "inner = t * g->T + h;                /* [T][H] */"),
    "page_first_lc_transposed": ("outer = (p * g->L + l) * g->C + c;   /* [P][L][C] */",
                                 "outer = (p * g->C + c) * g->L + l;   /* [P][L][C] */"),
    "layer_first_lc_transposed": ("outer = (l * g->C + c) * g->P + p;   /* [L][C][P] */",
                                  "outer = (c * g->L + l) * g->P + p;   /* [L][C][P] */"),
    "dev_inner_term_dropped": ("return (outer * (g->T * g->H) + inner) * g->B;\n}\n\n/* Byte offset of unit (slot",
                               "return (outer * (g->T * g->H)) * g->B;\n}\n\n/* Byte offset of unit (slot"),
    "host_lc_transposed": ("int64_t outer = (s * g->L + l) * g->C + c;   /* [S][L][C] */",
                           "int64_t outer = (s * g->C + c) * g->L + l;   /* [S][L][C] */"),
    "host_heads_flag_inverted": ("if (g->host_hnd)", "if (!g->host_hnd)"),
    "dev_heads_flag_inverted": ("if (g->dev_hnd)", "if (!g->dev_hnd)"),
    "order_flag_inverted": ("if (g->page_first)", "if (!g->page_first)"),
    "layer_range_one_too_many": ("(int64_t)layer + 1;", "(int64_t)layer + 2 > g->L ? g->L : (int64_t)layer + 2;"),
    "layer_range_skips_first": ("int64_t l_lo = layer < 0 ? 0 : layer;", "int64_t l_lo = layer < 0 ? 1 : layer;"),
    "short_copy": ("pool + kvo_dev_offset(g, src[i], l, c, t, h),\n                               (size_t)g->B);",
                   "pool + kvo_dev_offset(g, src[i], l, c, t, h),\n                               (size_t)g->B - 1);"),
    "backup_ids_swapped": ("host + kvo_host_offset(g, slot[i], l, c, t, h),\n                               pool + kvo_dev_offset(g, src[i]",
                           "host + kvo_host_offset(g, src[i], l, c, t, h),\n                               pool + kvo_dev_offset(g, slot[i]"),
    "restore_reads_dst_slot": ("host + kvo_host_offset(g, slot[i], l, c, t, h),\n                               (size_t)g->B);\n}",
                               "host + kvo_host_offset(g, dst[i], l, c, t, h),\n                               (size_t)g->B);\n}"),
    "offset_ignored": ("backup_range(g, pool_base + pool_offset, host", "backup_range(g, pool_base, host"),
    "thread_split_drops_items": ("job[k].i1 = n * (k + 1) / threads;", "job[k].i1 = n * (k + 1) / threads - (k == 0);"),
    "page_bytes_drops_C": ("return g->L * g->C * g->T * g->H * g->B;", "return g->L * g->T * g->H * g->B;"),
    "l3_put_indexes_file_by_slot": ("file[base + (int64_t)records[i] * rb + b] = host[(int64_t)slots[i] * rb + b];",
                                    "file[base + (int64_t)slots[i] * rb + b] = host[(int64_t)slots[i] * rb + b];"),
    "l3_get_drops_base": ("host[(int64_t)slots[i] * rb + b] = file[base + (int64_t)records[i] * rb + b];",
                          "host[(int64_t)slots[i] * rb + b] = file[(int64_t)records[i] * rb + b];"),
    "l3_put_short_record": ("for (int64_t b = 0; b < rb; ++b)\n            file[",
                            "for (int64_t b = 0; b < rb - 1; ++b)\n            file["),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, source, tmp_path):
    old, new = MUTATIONS[name]
    assert source.count(old) == 1, f"mutation anchor for {name} not unique in the oracle"
    mutated = source.replace(old, new)
    src = tmp_path / "kv_oracle_mut.c"
    src.write_text(mutated)
    so = tmp_path / "libkv_oracle_mut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", str(so),
                    str(src)], check=True)
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys\n"
        f"sys.path[:0] = [{os.path.dirname(here)!r}, {here!r}]\n"
        "import oracle, oracle_pins\n"
        f"lib = oracle.load({str(so)!r})\n"
        "tripped = []\n"
        "for pin in oracle_pins.ALL_PINS:\n"
        "    try:\n"
        "        pin(lib)\n"
        "    except AssertionError:\n"
        "        tripped.append(pin.__name__)\n"
        "print('TRIPPED', tripped)\n"
        "sys.exit(3 if tripped else 0)\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    # 3: a pin failed; negative: the mutant crashed on an out-of-bounds write
    assert r.returncode == 3 or r.returncode < 0, \
        f"no pin caught the planted mistake {name}: rc={r.returncode} {r.stdout[-300:]} {r.stderr[-300:]}"
