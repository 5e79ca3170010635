"""The README's Python example parses and calls only names the package exports."""
import ast
import os
import re

from tests._util import ROOT


def test_readme_example_uses_exported_names():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "README has no Python example"
    import eagle_tree_speculative_spec_gb300 as e3
    for code in blocks:
        tree = ast.parse(code)
        used = {n.attr for n in ast.walk(tree)
                if isinstance(n, ast.Attribute) and isinstance(n.value, ast.Name) and n.value.id == "e3"}
        assert used, "the example calls nothing from the package"
        for name in used:
            assert hasattr(e3, name), name
