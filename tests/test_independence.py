"""The oracle and the CUDA path share no code: no module of the product package imports the oracle
(or the tests), the oracle imports nothing of the product, and the only module both sides use is
the seeded input generator, which imports neither."""

import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    out = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            if node.level == 0 and node.module:
                out.add(node.module.split(".")[0])
    return out


def _py_files(d):
    for base, _, files in os.walk(os.path.join(ROOT, d)):
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(base, f)


def test_product_does_not_import_the_oracle():
    for f in _py_files("diffusion_transformer_gb300"):
        bad = _imports(f) & {"oracle", "tests", "dit_inputs"}
        assert not bad, (f, bad)


def test_oracle_does_not_import_the_product():
    for f in _py_files("oracle"):
        bad = _imports(f) & {"diffusion_transformer_gb300", "torch", "tests", "bench"}
        assert not bad, (f, bad)


def test_input_generator_imports_neither_side():
    bad = _imports(os.path.join(ROOT, "dit_inputs.py")) & {"oracle", "diffusion_transformer_gb300", "torch"}
    assert not bad, bad


def test_cuda_sources_reference_no_python_side():
    d = os.path.join(ROOT, "diffusion_transformer_gb300", "csrc")
    for f in os.listdir(d):
        src = open(os.path.join(d, f)).read()
        assert "oracle" not in src.lower(), f
