"""bench.py's host-side accounting on the CPU: the algorithmic bytes behind the roofline figure,
the source hash that keeps a committed DRAM-traffic capture tied to the kernel it measured, and
the clock-sample parsing behind the run's clock record."""
import os
import shutil

import numpy as np
import pytest
import torch

import bench
from decode_attention_compressed_gb300 import inputs as I
from oracle import zf_oracle as O
from tests import helpers as H


@pytest.fixture(scope="module")
def zf():
    return H.zf_module()


@pytest.mark.parametrize("name,kw", [("llama3_8b_batched", dict(batch=3, ctx=200, ctx_min=17)),
                                     ("long_ctx", dict(batch=2, ctx=300))])
def test_tile_bytes_counts_the_stored_records_of_the_context(zf, name, kw):
    """Per (request, kv head) the attention reads, for each 16-token tile holding context tokens,
    the K and V records of that tile: zf_page_head_bytes(16, compressed) twice for a compressed
    page head, the raw size twice for a raw one; plus q, the page table, lengths, out and lse."""
    w = I.scaled(I.WORKLOADS[name], **kw)
    layer = I.make_layer(w)
    oc = H.oracle_cache_from(layer, O)
    dirs = torch.from_numpy(oc.dir)
    comp16 = zf.lib().zf_page_head_bytes(16, 1)
    raw16 = zf.lib().zf_page_head_bytes(16, 0)
    P = w.page_size
    want = 0
    for b in range(w.batch):
        L = int(layer.seq_lens[b])
        for i in range(-(-L // P)):
            pid = int(layer.page_table[b, i])
            tiles = -(-min(P, L - i * P) // 16)
            for h in range(w.num_kv_heads):
                want += tiles * 2 * (comp16 if oc.dir[pid, h] == O.DIR_COMPRESSED else raw16)
    extras = (w.batch * w.num_q_heads * 128 * 2 + layer.page_table.numel() * 4 + w.batch * 4
              + w.batch * w.num_q_heads * (128 * 4 + 4))
    assert bench.tile_bytes(layer, dirs, compressed=True) == want + extras
    assert (oc.dir >= 0).any() and (oc.dir == O.DIR_COMPRESSED).any()
    dense = sum(-(-min(P, int(layer.seq_lens[b]) - i * P) // 16)
                for b in range(w.batch) for i in range(-(-int(layer.seq_lens[b]) // P))) * w.num_kv_heads * 2 * raw16
    assert bench.tile_bytes(layer, dirs, compressed=False) == dense + extras
    # ratio of dense to compressed bytes of a fully compressed context: 1024 / 784
    assert comp16 * 1024 == raw16 * 784


def _copy_sources(tmp_path):
    src = os.path.join(bench.ROOT, "decode_attention_compressed_gb300", "csrc")
    dst = tmp_path / "decode_attention_compressed_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(src, f), dst / f)
    return dst


def test_source_hash_ignores_comments_and_follows_code(tmp_path, monkeypatch):
    base = bench.kernel_source_hash()
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_source_hash() == base
    f = dst / bench.KERNEL_SOURCES[0]
    text = f.read_text()
    f.write_text("// a new comment line\n/* and a block\n comment */\n" + text.replace("\n", "\n\n", 5))
    assert bench.kernel_source_hash() == base
    f.write_text(text.replace("constexpr", "constexpr  int zf_extra_marker = 1; constexpr", 1))
    assert bench.kernel_source_hash() != base


def test_traffic_is_read_only_for_the_current_sources(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    h = bench.kernel_source_hash()
    (tmp_path / "profiles" / "attn_kernel_dram_traffic_by_workload.txt").write_text(
        "# workload launches bytes hash\n"
        f"wl_a 3 123456 {h}\n"
        "wl_b 3 999 0000000000000000\n")
    assert bench.read_traffic("wl_a") == 123456.0
    assert bench.read_traffic("wl_b") is None          # captured on other kernel code
    assert bench.read_traffic("wl_c") is None


def test_clock_summary_from_nvidia_smi_lines(tmp_path):
    s = bench.ClockSampler(0)
    s.nvml = None
    s.proc = object()
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 2070, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n")
        f.write("garbage line\n")
    out = s.summary()
    assert out["source"] == "nvidia-smi" and out["samples"] == 3
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(s.path)



def test_multi_token_lines_name_real_workloads_and_wide_column_sets():
    """The default run's multi_token object times shapes whose columns per kv head (query heads per
    kv head x new tokens) take the tensor-memory kernel (more than 8)."""
    from decode_attention_compressed_gb300 import inputs as I
    assert bench.MULTI_TOKEN
    for name, T in bench.MULTI_TOKEN:
        w = I.WORKLOADS[name]
        assert T > 1 and w.num_q_heads // w.num_kv_heads * T > 8


@pytest.mark.parametrize("tokens", [1, 3])
def test_reference_arm_line_has_this_arms_config(tokens, monkeypatch):
    """The reference arm (the oracle on the host cores) prints the same `config` object as this
    library's arm for the same arguments, so the two lines compare like for like; with several new
    tokens per request its sample runs the multi-token oracle."""
    monkeypatch.setattr(bench, "usable_cores", lambda: 2)
    args = bench.argparse.Namespace(workload="tiny", layers=None, batch=None, steps=1, warmup=3,
                                    tokens=tokens, kernel="auto")
    res = bench.run_reference(args, 0)
    w = bench.workload_of(args)
    assert res["config"] == bench.arm_config(w, tokens, "auto", 1)
    assert res["impl"] == "reference" and res["extrapolated"] is True
    assert f"{tokens} new token" in res["cpu_baseline"]["sample"]
    assert res["value"] > 0 and res["e2e"]["value"] == res["value"]
    assert bench.run_reference(args, 1) is None          # only rank 0 runs it


def test_l2_note_follows_the_smallest_step():
    big = bench.arm_config(I.WORKLOADS["llama7b_mha_8192"], 1, "auto", 1)["l2"]
    small = bench.arm_config(I.WORKLOADS["tiny"], 1, "auto", 1)["l2"]
    assert "at least 3.29 GB" in big and "> 129 MiB L2" in big
    assert "may stay in the 129 MiB L2" in small
