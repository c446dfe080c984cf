"""bench.py's roofline traffic figures: the committed ncu summary is read only
while the captured kernel's sources are the ones it was taken on, so a changed
kernel reports no traffic rather than a stale figure."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _copy_tree(tmp):
    dst = os.path.join(tmp, "repo")
    os.makedirs(os.path.join(dst, "gqa_decoder_forward_gb300"))
    shutil.copytree(os.path.join(ROOT, "profiles"), os.path.join(dst, "profiles"))
    shutil.copytree(os.path.join(ROOT, "gqa_decoder_forward_gb300", "csrc"),
                    os.path.join(dst, "gqa_decoder_forward_gb300", "csrc"),
                    ignore=shutil.ignore_patterns("*.o"))
    return dst


def test_traffic_is_read_while_sources_match(tmp_path, monkeypatch):
    dst = _copy_tree(str(tmp_path))
    monkeypatch.setattr(bench, "ROOT", dst)
    for kernel in ("decode_step_persistent", "gemm_gate_up_swiglu"):
        got = bench.ncu_traffic(kernel)
        assert isinstance(got, int) and got > 0, kernel


def test_traffic_is_dropped_once_a_source_changes(tmp_path, monkeypatch):
    dst = _copy_tree(str(tmp_path))
    monkeypatch.setattr(bench, "ROOT", dst)
    with open(os.path.join(dst, "gqa_decoder_forward_gb300", "csrc", "matvec_core.cuh"), "a") as fh:
        fh.write("\n// changed\n")
    assert bench.ncu_traffic("decode_step_persistent") is None
    # a kernel whose sources did not change keeps its figure
    assert isinstance(bench.ncu_traffic("gemm_gate_up_swiglu"), int)


def test_traffic_of_an_unknown_kernel_or_missing_summary_is_none(tmp_path, monkeypatch):
    dst = _copy_tree(str(tmp_path))
    monkeypatch.setattr(bench, "ROOT", dst)
    assert bench.ncu_traffic("no_such_kernel") is None
    os.remove(os.path.join(dst, "profiles", "ncu_traffic.md"))
    assert bench.ncu_traffic("decode_step_persistent") is None


def test_reference_arm_states_the_oracle_weight_bytes():
    # 52 layers of 1,181,773,824 B plus the embedding table and lm_head (2 x 166,912 x 7,168 x 2 B)
    assert abs(bench.oracle_weight_gb(52) - (52 * 1_181_773_824 + 2 * 166_912 * 7_168 * 2) / 1e9) < 1e-9
    assert bench.host_ram_gb() > 0
