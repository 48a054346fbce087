"""Host-side arithmetic of bench.py, on CPU: the algorithmic FLOP and byte counts behind every
reported rate, the roofline fraction, and the rule that a profile summary's traffic is used
only while its source hash matches the kernel sources."""
import torch

import bench
import workloads


def test_causal_pairs_closed_form():
    # bottom-right causal: query i sees Lkv - Lq + i + 1 keys (all of them once that exceeds Lkv)
    for Lq, Lkv in ((512, 16384), (64, 64), (7, 100), (300, 40)):
        want = sum(min(Lkv, max(0, Lkv - Lq + i + 1)) for i in range(Lq))
        assert workloads.causal_pairs(Lq, Lkv) == want
    assert workloads.causal_pairs(512, 16384) == 512 * (16384 - 512) + 512 * 513 // 2


def test_headline_flops():
    c = workloads.gqa_prefill_chunk()
    pairs = 512 * (16384 - 512) + 512 * 513 // 2
    assert bench.prefill_flops(c) == 4.0 * 128 * 32 * pairs == 135295664128.0


def test_decode_bytes_count_each_kv_byte_once():
    c = workloads.PagedCase(B=3, Hq=8, Hkv=2, D=64, page_size=16, num_pages=64, min_len=1,
                            max_len=300, seq_lens=[1, 129, 300])
    lens = torch.tensor([1, 129, 300], dtype=torch.int32)
    b = bench.decode_bytes(c, lens)
    assert b["kv"] == (1 + 129 + 300) * 2 * 64 * 2 * 2          # K and V, every kv head
    pages = (1 + 9 + 19) * 4                                    # one int32 page id per page
    q = 3 * 8 * 64 * 2
    assert b["kernel"] == b["kv"] + pages + q + 3 * 4
    assert b["total"] == b["kernel"] + 3 * 8 * 64 * 2 + 3 * 8 * 4  # + out and lse


def test_mla_bytes_count_ckv_and_kpe_once():
    c = workloads.MlaCase(B=2, H=64, seq_len=None, seq_lens=[100, 33])
    b = bench.mla_bytes(c)
    assert b["kv"] == 133 * (512 + 64) * 2
    assert b["total"] - b["kernel"] == 2 * 64 * 512 * 2 + 2 * 64 * 4


def test_roofline_fraction():
    pk = {"source": "measured"}
    r = bench.roofline("hbm", 5000.0, 6692.1, "GB/s", None, pk)
    assert r["frac"] == round(5000.0 / 6692.1, 4) and r["peak_source"] == "measured (copy)"
    r = bench.roofline("tensor", 1000.0, 1941.8, "TFLOP/s", 123, pk)
    assert r["traffic"] == 123 and r["peak_source"] == "measured (burst)"


def test_profile_traffic_only_while_sources_match(tmp_path, monkeypatch):
    csrc = tmp_path / "softmax_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES["decode"]:
        (csrc / name).write_text(f"// {name}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.src_hash("decode")
    (tmp_path / "profiles" / "p.md").write_text(
        f"source_sha256: {h}\ntraffic_bytes_per_launch: 4242\n")
    assert bench.profiled_traffic("p.md", "decode") == 4242
    (csrc / "decode.cu").write_text("// decode.cu, edited\n")
    assert bench.profiled_traffic("p.md", "decode") is None      # stale: no traffic
    assert bench.profiled_traffic("absent.md", "decode") is None
