"""CPU checks of the sources the library embeds for run-time compilation:
every file the forward kernel header includes is embedded under its include
name, verbatim, and none of them contains the raw-string delimiter."""
import os
import re
import tempfile

from attention_residuals_gb300 import build


def test_embedded_sources_are_verbatim_and_complete():
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "attnres_jit_sources.inc")
        build._write_jit_sources(path)
        text = open(path).read()
    embedded = dict(re.findall(r'\{"([^"]+)", R"ATTNRES_SRC\((.*?)\)ATTNRES_SRC"\}', text, flags=re.S))
    for name, folder in build.JIT_FILES:
        with open(os.path.join(folder, name)) as f:
            assert embedded[name] == f.read(), name
    # every quoted include of the embedded files is itself embedded
    for name, body in embedded.items():
        for inc in re.findall(r'#include\s+"([^"]+)"', body):
            assert inc in embedded, (name, inc)
