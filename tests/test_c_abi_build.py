"""The C ABI from C (no GPU needed): tests/c_abi_client.c, a plain C99
client, compiles with -Wall -Wextra -Werror against include/attnbwd.h and
links against the library, so every call it makes is exported."""
import os

from c_client_build import build_client


def test_c_client_compiles_and_links(tmp_path):
    exe = build_client(str(tmp_path / "c_abi_client"))
    assert os.path.exists(exe)
