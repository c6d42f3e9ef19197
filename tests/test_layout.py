"""Separation rules the parity claims rest on, checked on the source tree: the product package
never reaches the oracle (test infrastructure only), the oracle's C shares no header with the
CUDA path, and no source reads a scratch folder."""
import ast
import pathlib
import re

ROOT = pathlib.Path(__file__).resolve().parent.parent
PKG = ROOT / "block_scaled_mxfp4_bf16_gb300"
ORACLE = ROOT / "oracle"
SOURCE_DIRS = (PKG, ORACLE, ROOT / "tests", ROOT / "include")   # plus the scripts at the root


def _sources(base: pathlib.Path, suffixes):
    for p in base.rglob("*"):
        if p.suffix in suffixes and p.is_file() and "__pycache__" not in p.parts:
            yield p


def _all_sources(suffixes):
    for d in SOURCE_DIRS:
        yield from _sources(d, suffixes)
    yield from (p for p in ROOT.glob("*") if p.suffix in suffixes and p.is_file())


def _imported_modules(py: pathlib.Path):
    for node in ast.walk(ast.parse(py.read_text())):
        if isinstance(node, ast.Import):
            yield from (a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            yield node.module or ""


def test_product_package_never_imports_the_oracle():
    for py in _sources(PKG, {".py"}):
        for mod in _imported_modules(py):
            assert mod != "oracle" and not mod.startswith("oracle."), f"{py} imports {mod}"


def test_cuda_sources_name_no_oracle_symbol():
    for src in _sources(PKG, {".cu", ".cuh", ".h", ".c", ".cpp"}):
        text = src.read_text()
        assert "oracle_" not in text and "mxfp4_oracle" not in text, src


def test_oracle_c_includes_only_system_headers():
    for src in _sources(ORACLE, {".c", ".h"}):
        for line in src.read_text().splitlines():
            m = re.match(r'\s*#\s*include\s*(\S+)', line)
            if m:
                assert m.group(1).startswith("<"), f"{src}: {line.strip()}"


def test_no_source_reads_the_scratch_folder():
    pat = re.compile(r"""(["'/\\])_work(/|\\|["'])""")
    this = pathlib.Path(__file__).resolve()   # names the folder only to look for it
    for src in _all_sources({".py", ".cu", ".cuh", ".h", ".c", ".cpp", ".sh", ".toml", ".cfg", ".ini"}):
        if src.resolve() != this:
            assert not pat.search(src.read_text()), src
