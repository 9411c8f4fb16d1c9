"""The pins of ``oracle/heads.py`` must catch plausible mistakes (CPU only).

Each case plants one mistake in a private copy of the oracle package (a
wrong rounding direction, a wrong format constant, swapped operands, an
off-by-one rank, an ignored index), then runs the pins of that module in a
subprocess whose ``import oracle`` finds the copy.  Every planted mistake must
make at least one pin fail.

Which pin catches which mistake (first failing test, as last observed):

* E4M3 ties to odd codes -- ``test_e4m3_encode_matches_library_conversion``
* E4M3 maximum of another format -- ``test_e4m3_encode_matches_library_conversion``
* E4M3 subnormal scale -- ``test_e4m3_decode_known_codes``
* SiLU applied to the up half -- ``test_swiglu_quant_row_maximum_maps_to_448_and_error_bound``
* sigmoid sign -- ``test_swiglu_quant_row_maximum_maps_to_448_and_error_bound``
* scale inverted -- ``test_swiglu_quant_row_maximum_maps_to_448_and_error_bound``
* first row of a sequence instead of its last -- ``test_label_scores_match_library_and_closed_forms``
* stop candidates finished up to rank W inclusive -- ``test_split_finished_hand_example``
* history not gathered by parent -- ``test_reorder_history_hand_example``
* followed beams scored with the normaliser's sign flipped -- ``test_following_its_own_beams_changes_nothing``
"""
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MISTAKES = {
    "E4M3 ties to odd codes": ("((dhi == dlo) & (_POS_CODES[hi] % 2 == 0))",
                               "((dhi == dlo) & (_POS_CODES[hi] % 2 == 1))"),
    "E4M3 maximum of another format": ("E4M3_MAX = 448.0", "E4M3_MAX = 240.0"),
    "E4M3 subnormal scale": ("m / 8.0 * 2.0 ** -6", "m / 8.0 * 2.0 ** -7"),
    "SiLU applied to the up half": ("g, u = gu[:, :I], gu[:, I:]", "u, g = gu[:, :I], gu[:, I:]"),
    "sigmoid sign": ("g / (1.0 + np.exp(-g)) * u", "g / (1.0 + np.exp(g)) * u"),
    "scale inverted": ("_f32(amax / E4M3_MAX)", "_f32(E4M3_MAX / np.where(amax > 0, amax, 1.0))"),
    "first row of a sequence instead of its last": ("np.dot(h[s1 - 1], w[k])", "np.dot(h[s0], w[k])"),
    "stop candidates finished up to rank W inclusive": ("if rank < W:", "if rank <= W:"),
    "history not gathered by parent": ("out[b, :t] = np.asarray(hist_in)[p, :t]",
                                       "out[b, :t] = np.asarray(hist_in)[b, :t]"),
    "followed beams scored with the normaliser's sign flipped": (
        "lp = (x - np.asarray(lse, dtype=np.float32)[par]).astype(np.float32)",
        "lp = (x + np.asarray(lse, dtype=np.float32)[par]).astype(np.float32)"),
}

PIN_FILES = ["test_oracle_heads.py", "test_oracle_loop.py"]


def _copy_tree(dst):
    """The parts of the repository the pins import: the oracle package (the
    mutated copy), the input generators, and the pin files with their conftest."""
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    pkg = os.path.join(dst, "attention_packed_varlen_gb300")
    os.makedirs(pkg)
    open(os.path.join(pkg, "__init__.py"), "w").close()
    shutil.copy(os.path.join(ROOT, "attention_packed_varlen_gb300", "workloads.py"), pkg)
    os.makedirs(os.path.join(dst, "tests"))
    for f in ["__init__.py", "conftest.py"] + PIN_FILES:
        src = os.path.join(HERE, f)
        if os.path.exists(src):
            shutil.copy(src, os.path.join(dst, "tests"))


def _run_pins(tmp_path):
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider"]
                          + [str(tmp_path / "tests" / f) for f in PIN_FILES],
                          env=env, cwd=str(tmp_path), capture_output=True, text=True, timeout=600)


def test_unmutated_copy_passes(tmp_path):
    # the harness itself: the copied package passes its pins unchanged, so a
    # failure below comes from the planted mistake, not from the copy
    _copy_tree(tmp_path)
    r = _run_pins(tmp_path)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MISTAKES))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MISTAKES[name]
    _copy_tree(tmp_path)
    path = tmp_path / "oracle" / "heads.py"
    src = path.read_text()
    assert src.count(old) == 1, f"mutation anchor for '{name}' not found exactly once"
    path.write_text(src.replace(old, new))
    r = _run_pins(tmp_path)
    assert r.returncode == 1, f"planted mistake '{name}' passed every pin (rc {r.returncode}):\n{r.stdout[-2000:]}"
    assert " failed" in r.stdout, r.stdout[-2000:]
