"""Static rules on the CUDA sources (CPU only).

- Under programmatic dependent launch a kernel starts while its predecessor may still run, and
  the non-coherent load path (`__ldg`, ld.global.nc) requires its data to stay unchanged for the
  reading kernel's whole lifetime. So `__ldg` may only read buffers that no kernel of the library
  writes: the step's inputs (indexer and attention queries, head weights, visible lengths, window
  rows, the writer's latents, gates, W_idx and entry offsets). The cache, the pool, the top-k
  lists and the workspace are other kernels' outputs and must be read with coherent loads.
- No source uses a cluster-multicast copy: every CTA loads its own tiles, the form the
  one-process-per-GPU replica mode keeps to.
"""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "hierarchical_sparse_attention_index_gb300", "csrc")

# buffers no kernel of the library writes
INPUTS = ("p.vis", "p.swa", "p.wkv", "p.wgate", "p.w_idx", "p.start_entry", "q16x128", "w16")
# buffers written by a kernel of the library
OUTPUTS = ("kv_q", "kv_s", "ik_q", "ik_s", "pool", "topk", "scores", "blkmax", "hist", "cand", "part", "ws")


def sources():
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, name), encoding="utf-8") as f:
                yield name, f.read().splitlines()


def ldg_argument(line):
    start = line.index("__ldg(") + len("__ldg(")
    depth, out = 1, []
    for ch in line[start:]:
        depth += ch == "("
        depth -= ch == ")"
        if depth == 0:
            break
        out.append(ch)
    return "".join(out)


def source_of(lines, i, name):
    """The right-hand side that defines local pointer `name`, searching back from line i."""
    pat = re.compile(r"\b" + re.escape(name) + r"\s*=")
    for j in range(i, max(-1, i - 40), -1):
        if pat.search(lines[j]):
            return " ".join(lines[j:j + 3])
    return ""


def test_non_coherent_loads_read_only_step_inputs():
    seen = 0
    for name, lines in sources():
        for i, line in enumerate(lines):
            if "__ldg(" not in line or line.lstrip().startswith("//"):
                continue
            seen += 1
            arg = ldg_argument(line)
            if any(inp in arg for inp in INPUTS):
                continue
            base = re.match(r"\s*(?:reinterpret_cast<[^>]*>\()?\s*([A-Za-z_]\w*)", arg)
            assert base, f"{name}:{i + 1}: cannot read the __ldg argument {arg!r}"
            definition = source_of(lines, i, base.group(1))
            assert any(inp in definition for inp in INPUTS), (
                f"{name}:{i + 1}: __ldg reads {arg!r}, which is not a step input "
                f"(defined as {definition.strip()!r})")
            assert not any(re.search(r"\b" + o + r"\b", definition) for o in OUTPUTS), f"{name}:{i + 1}"
    assert seen > 0


def test_no_cluster_multicast_copies():
    for name, lines in sources():
        assert "multicast::cluster" not in "\n".join(lines), f"{name} uses a cluster-multicast copy"
