"""Host logic of bench.py that its reported numbers depend on (CPU only)."""
import shutil

import bench


def test_traffic_key_ignores_comments_and_layout_not_code(tmp_path, monkeypatch):
    """The committed ncu traffic figures are keyed on the kernel code: a comment
    or a change of layout keeps the key, any change of code voids it (the bench
    then reports traffic null)."""
    src = tmp_path / "csrc"
    shutil.copytree(bench.CSRC, src)
    monkeypatch.setattr(bench, "CSRC", str(src))
    h0 = bench.kernel_source_hash()
    f = src / "ss_scan1d.cuh"
    text = f.read_text()
    f.write_text("// a new comment line\n/* and a block\n   comment */\n" +
                 text.replace("\n", "\n\n  ", 40))
    assert bench.kernel_source_hash() == h0
    f.write_text(text.replace("float", "double", 1))
    assert bench.kernel_source_hash() != h0


def test_traffic_lookup_is_null_off_key(tmp_path, monkeypatch):
    """A traffic table recorded under another key yields no figure."""
    table = tmp_path / "ncu_traffic.json"
    table.write_text('{"source_hash": "0000000000000000", "workloads": '
                     '{"mamba130m_layer_b8_d1536_l2048_n16": {"dram_bytes_per_launch": 1}}}')
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(table))
    assert bench.ncu_traffic_named("mamba130m_layer_b8_d1536_l2048_n16") is None
    key = bench.kernel_source_hash()
    table.write_text('{"source_hash": "%s", "workloads": '
                     '{"mamba130m_layer_b8_d1536_l2048_n16": {"dram_bytes_per_launch": 1}}}' % key)
    assert bench.ncu_traffic_named("mamba130m_layer_b8_d1536_l2048_n16") == 1
