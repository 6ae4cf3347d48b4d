"""Constants of the CUDA kernels, read from their source files, so that the
host models of the kernels' synchronisation run with the stage counts, warp
roles and barrier arrival counts the kernels are compiled with (a change in a
kernel changes the model's run, or fails the read, instead of leaving the
model behind)."""
import ast
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "..", "block_sparse_attention_08_gb300", "csrc")


def _source(file):
    with open(os.path.join(CSRC, file)) as f:
        return f.read()


def _eval(expr, file, depth=0):
    """Integer value of a constant expression of literals, + - * / ( ) and
    other constexpr names of `file` (or of common.cuh)."""
    tree = ast.parse(expr.strip(), mode="eval")

    def ev(n):
        if isinstance(n, ast.Expression):
            return ev(n.body)
        if isinstance(n, ast.Constant) and isinstance(n.value, int):
            return n.value
        if isinstance(n, ast.BinOp) and isinstance(n.op, (ast.Add, ast.Sub, ast.Mult, ast.Div, ast.FloorDiv)):
            a, b = ev(n.left), ev(n.right)
            if isinstance(n.op, ast.Add):
                return a + b
            if isinstance(n.op, ast.Sub):
                return a - b
            if isinstance(n.op, ast.Mult):
                return a * b
            return a // b  # C++ integer division of non-negative values
        if isinstance(n, ast.Name):
            assert depth < 8, expr
            return kconst(n.id, file, depth + 1)
        raise ValueError(f"unsupported expression in {file}: {expr}")
    return ev(tree)


def kconst(name, file, depth=0):
    """Value of `constexpr int <name> = ...;` in csrc/<file> (then common.cuh)."""
    for f in (file, "common.cuh"):
        m = re.search(r"constexpr\s+(?:int|size_t|uint32_t)\s+" + re.escape(name) + r"\s*=\s*([^;,]+)[;,]", _source(f))
        if m:
            return _eval(m.group(1), f, depth)
    raise KeyError(f"{name} not found in {file} or common.cuh")


def mbar_count(barrier, file, after=None):
    """Arrival count of the first `mbar_init(&sm.<barrier>..., <count>)` in
    csrc/<file> (the first one after the text `after`, when given)."""
    text = _source(file)
    start = text.index(after) if after else 0
    m = re.compile(r"mbar_init\(&sm\." + re.escape(barrier) + r"(?:\[[^\]]*\])?\s*,\s*([^)]+)\)").search(text, start)
    if not m:
        raise KeyError(f"mbar_init of {barrier} not found in {file}")
    return _eval(m.group(1), file)
