"""The tuned launch-choice table: parsing, matching, folder loading and the
override reaching the plan (visible on the host through the workspace size,
which grows with the token tile and the K split)."""
import os

import pytest

from lora_mixture_experts_gb300 import binding
from lora_mixture_experts_gb300.binding import MoeLoraError, moelora_dims, moelora_linear_dims

DEC = moelora_dims(16, 4, 32, 2880, 2880, 8, 32)


@pytest.fixture(autouse=True)
def clear_table(lib):
    binding.moelora_load_tuning(None)
    yield
    binding.moelora_load_tuning(None)


def _write(tmp_path, name, text):
    p = tmp_path / name
    p.write_text(text)
    return str(p)


def test_override_changes_the_plan(tmp_path):
    base = binding.moelora_workspace_bytes(DEC)
    binding.moelora_load_tuning(_write(tmp_path, "a.cfg", "moe T=1-64 E=32 ksplit=1   # one split\n"))
    assert binding.moelora_tuning_entries() == 1
    ks1 = binding.moelora_workspace_bytes(DEC)
    binding.moelora_load_tuning(_write(tmp_path, "b.cfg", "moe T=16 k=4 E=32 H=2880 I=2880 L=8 r=32 ksplit=4\n"))
    ks4 = binding.moelora_workspace_bytes(DEC)
    assert ks1 < base < ks4                     # the default splits the decode down phase in two
    binding.moelora_load_tuning(_write(tmp_path, "c.cfg", "moe T=16 tn=256\n"))
    assert binding.moelora_workspace_bytes(DEC) > base   # wider token tiles: bigger shrink buffers


def test_non_matching_lines_are_ignored(tmp_path):
    base = binding.moelora_workspace_bytes(DEC)
    binding.moelora_load_tuning(_write(tmp_path, "a.cfg", "moe T=17-99 ksplit=4\nmoe E=64 ksplit=4\nlinear ksplit=4\n"))
    assert binding.moelora_tuning_entries() == 3
    assert binding.moelora_workspace_bytes(DEC) == base


def test_first_match_wins_and_linear_entries(tmp_path):
    binding.moelora_load_tuning(_write(tmp_path, "a.cfg", "moe ksplit=1\nmoe ksplit=4\n"))
    one = binding.moelora_workspace_bytes(DEC)
    binding.moelora_load_tuning(_write(tmp_path, "b.cfg", "moe ksplit=1\n"))
    assert binding.moelora_workspace_bytes(DEC) == one
    lin = moelora_linear_dims(8, 8192, 28672, 32, 16)
    base = binding.moelora_linear_workspace_bytes(lin)
    binding.moelora_load_tuning(_write(tmp_path, "c.cfg", "linear T=1-64 K=8192 N=28672 ksplit=1\n"))
    assert binding.moelora_linear_workspace_bytes(lin) < base      # no fp32 split partials


def test_folder_loads_every_cfg_in_name_order(tmp_path):
    d = tmp_path / "tuned"
    d.mkdir()
    (d / "b.cfg").write_text("moe ksplit=4\n")
    (d / "a.cfg").write_text("# tuned on GB300\nmoe ksplit=1\n\n")
    (d / "notes.txt").write_text("moe ksplit=3\n")
    binding.moelora_load_tuning(str(d))
    assert binding.moelora_tuning_entries() == 2
    only1 = binding.moelora_workspace_bytes(DEC)
    binding.moelora_load_tuning(_write(tmp_path, "x.cfg", "moe ksplit=1\n"))
    assert binding.moelora_workspace_bytes(DEC) == only1         # a.cfg came first


@pytest.mark.parametrize("text", ["moe tn=48\n", "moe ksplit=9\n", "attention T=4\n", "moe T=9-3\n", "moe bogus=1\n",
                                  "moe T\n", "moe T=x\n", "moe T=5x\n", "moe T=-3\n", "moe T=4-\n", "moe k=4q\n",
                                  "moe phases=3\n", "moe phases=0\n"])
def test_malformed_tables_are_rejected_and_keep_the_old_one(tmp_path, text):
    binding.moelora_load_tuning(_write(tmp_path, "ok.cfg", "moe ksplit=1\n"))
    with pytest.raises(MoeLoraError):
        binding.moelora_load_tuning(_write(tmp_path, "bad.cfg", text))
    assert binding.moelora_tuning_entries() == 1
    with pytest.raises(MoeLoraError):
        binding.moelora_load_tuning(str(tmp_path / "missing.cfg"))


def test_shipped_table_parses():
    path = os.path.join(os.path.dirname(binding.__file__), "tuning")
    if not os.path.isdir(path):
        pytest.skip("no shipped table")
    binding.moelora_load_tuning(path)
    assert binding.moelora_tuning_entries() > 0


def test_sweep_buckets_cover_every_batch_size():
    from lora_mixture_experts_gb300 import tune
    for fam in tune.FAMILIES.values():
        b = tune.buckets(fam.ladder)
        assert b[0][0] == 1 and b[-1][1] == tune.T_MAX
        for (lo, hi), t in zip(b, fam.ladder):
            assert lo <= t <= hi                      # each sampled size sits in its own bucket
        for (_, hi), (lo, _) in zip(b, b[1:]):
            assert lo == hi + 1                       # no gaps, no overlaps


def test_sweep_lines_merge_buckets_and_load(tmp_path):
    from lora_mixture_experts_gb300 import tune
    key = "moe T=@ k=4 E=32 H=2880 I=2880 L=8 r=32"
    picks = [(1, 1, "tn=16 ksplit=2 phases=2"), (2, 2, "tn=16 ksplit=2 phases=2"),
             (3, 5, None), (6, 11, "tn=32 ksplit=1 phases=2"), (12, tune.T_MAX, "tn=256 ksplit=1")]
    lines = tune.merge_lines(key, picks)
    assert lines == ["moe T=1-2 k=4 E=32 H=2880 I=2880 L=8 r=32 tn=16 ksplit=2 phases=2",
                     "moe T=6-11 k=4 E=32 H=2880 I=2880 L=8 r=32 tn=32 ksplit=1 phases=2",
                     f"moe T=12-{tune.T_MAX} k=4 E=32 H=2880 I=2880 L=8 r=32 tn=256 ksplit=1"]
    binding.moelora_load_tuning(_write(tmp_path, "s.cfg", "\n".join(lines) + "\n"))
    assert binding.moelora_tuning_entries() == 3
    # T = 4 falls in the built-in bucket, T = 8 (off the ladder) in the tn=32 one
    base = binding.moelora_workspace_bytes(moelora_dims(8, 4, 32, 2880, 2880, 8, 32))
    binding.moelora_load_tuning(None)
    assert binding.moelora_workspace_bytes(moelora_dims(8, 4, 32, 2880, 2880, 8, 32)) != base


def test_gate_up_split_key(tmp_path):
    # a one-expert layer: guksplit plans the gate_up phase's fp32 parts
    # (visible as a larger workspace); out-of-range values are rejected
    mlp = moelora_dims(8, 1, 1, 8192, 14336, 32, 16)
    base = binding.moelora_workspace_bytes(mlp)
    binding.moelora_load_tuning(_write(tmp_path, "g.cfg", "moe T=1-22 E=1 tn=16 guksplit=2\n"))
    assert binding.moelora_workspace_bytes(mlp) > base
    with pytest.raises(MoeLoraError):
        binding.moelora_load_tuning(_write(tmp_path, "bad.cfg", "moe T=8 guksplit=5\n"))
    # CTA-pair tiles keep one gate_up split
    binding.moelora_load_tuning(_write(tmp_path, "p.cfg", "moe T=1-22 E=1 tn=256 guksplit=2\n"))
    w256 = binding.moelora_workspace_bytes(mlp)
    binding.moelora_load_tuning(_write(tmp_path, "q.cfg", "moe T=1-22 E=1 tn=256\n"))
    assert binding.moelora_workspace_bytes(mlp) == w256
