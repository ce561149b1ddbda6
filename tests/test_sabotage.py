"""Separating arms: every pin that guards a rule of the profile must fail when
that rule is broken.

The pages count a numerical test as evidence only once a separating arm shows
that it fails when the rule it guards is broken ("mojolearn" PyPI page,
section "Development"; the home page speaks of stage-level identity cards and
sabotage tests). Each arm below is the oracle's own C source built with one
SABOTAGE_* define, which plants one plausible mistake (det_oracle.c holds the
blocks; the shipped oracle defines none). For each arm the named pins run in a
child pytest process against that build (DET_ORACLE_LIB), and at least one of
them must fail. The same pins pass against the shipped oracle in the main run.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

G = "tests/test_oracle_gemm.py::"
E = "tests/test_oracle_exp_log_steps.py::"
R = "tests/test_oracle_rowops.py::"
B = "tests/test_oracle_rmsnorm_bwd.py::"
S = "tests/test_oracle_shardsum.py::"
A = "tests/test_oracle_expl_adamw.py::"

# define -> (the rule it breaks, the pins that must catch it)
ARMS = {
    "SABOTAGE_CHUNK128": ("GEMM chunks 256 wide (R3)", [G + "test_chunk_width_256"]),
    "SABOTAGE_CHUNK_REVERSED": ("chunk partials added left to right (R2)",
                                [G + "test_chunks_summed_left_to_right"]),
    "SABOTAGE_FIRST_PRODUCT_SEED": ("chains start at +0 (R1)",
                                    [G + "test_chain_starts_at_plus_zero"]),
    "SABOTAGE_ROUNDF": ("exp's n rounds half to even (R14 tie rule)",
                        [E + "test_exp_ties_of_the_rounding_step"]),
    "SABOTAGE_EXP_LN2_SPLIT": ("exp's ln 2 split (R14)",
                               [E + "test_exp_reduction_sensitive_arguments"]),
    "SABOTAGE_EXP_HORNER_UNFUSED": ("exp's Horner steps by fmaf (R14)",
                                    [E + "test_exp_every_binade_stratified"]),
    "SABOTAGE_CONTRACT_LOG": ("log's h - s(h + R) rounded twice (R15)",
                              [E + "test_log_every_binade_both_sides_of_the_split"]),
    "SABOTAGE_RECIP_D": ("RMSNorm divides by D (R8)", [R + "test_rmsnorm_exact_emulation_tiny"]),
    "SABOTAGE_BUTTERFLY_ORDER": ("butterfly offsets 16, 8, 4, 2, 1 (R6)",
                                 [R + "test_rmsnorm_butterfly_pinned"]),
    "SABOTAGE_ELEMENT_OWNERSHIP": ("chains own groups of 4 (R6)",
                                   [R + "test_rmsnorm_chain_ownership_pinned"]),
    "SABOTAGE_XENT_LANES32": ("cross-entropy over 256 chains (R10)",
                              [R + "test_xent_tree_restated"]),
    "SABOTAGE_CONTRACT_RMSBWD": ("dx's h - xhat q rounded twice (R22)",
                                 [B + "test_exact_emulation_tiny"]),
    "SABOTAGE_ONE_CHAIN_DGAIN": ("dgain in 256-row chunks (R23)",
                                 [B + "test_dgain_chunks_pinned"]),
    "SABOTAGE_SHARD_REVERSED": ("shard gradients summed left to right (R25)",
                                [S + "test_left_to_right_pinned"]),
    "SABOTAGE_ADAMW_RECIP_BC": ("AdamW divides by the corrections (R18)",
                                [A + "test_adamw_exact_emulation_elementwise"]),
}


def run_arm(define, pins, workdir):
    lib = oracle.build_variant([define], os.path.join(workdir, f"lib_{define}.so"))
    env = dict(os.environ, DET_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu", *pins], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    return r.returncode, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    work = str(tmp_path_factory.mktemp("arms"))
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {d: ex.submit(run_arm, d, pins, work) for d, (_, pins) in ARMS.items()}
        return {d: f.result() for d, f in futs.items()}


@pytest.mark.parametrize("define", sorted(ARMS))
def test_arm_fails_a_named_pin(results, define):
    rc, out = results[define]
    rule, pins = ARMS[define]
    # pytest exits 1 when tests ran and some failed (2-5: errors, none collected)
    assert rc == 1 and " failed" in out, f"{define} ({rule}) passed {pins}:\n{out}"


def test_the_shipped_oracle_defines_no_arm():
    src = open(os.path.join(ROOT, "oracle", "det_oracle.c")).read()
    for d in ARMS:
        assert f"#ifdef {d}" in src or f"#ifndef {d}" in src, d
        assert f"#define {d}" not in src, d
    assert not any(f.startswith("-DSABOTAGE") for f in oracle.CFLAGS)
