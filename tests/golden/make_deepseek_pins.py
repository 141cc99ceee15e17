"""Writes pretoken_pins_deepseek.txt: split examples for the DeepSeek-style
pattern, produced by the third-party `regex` module from the pattern text
(the same text include/tok.h and oracle/pretokenize.py state).  The oracle is
checked against these; nothing here calls the oracle or the library.

Run where `regex` is installed:  python tests/golden/make_deepseek_pins.py
"""
import json
import os

import regex

CJK = r"[\p{scx=Han}\p{scx=Hiragana}\p{scx=Katakana}\p{scx=Hangul}]"
DEEPSEEK_RE = (r"(?i:'s|'t|'re|'ve|'m|'ll|'d)|[^\r\n\p{L}\p{N}]?(?:(?!" + CJK + r")\p{L})+|(?:(?=" + CJK
               + r")\p{L})+|\p{N}{1,3}| ?[^\s\p{L}\p{N}]+[\r\n]*|\s*[\r\n]+|\s+(?!\S)|\s+")

EXAMPLES = [
    "中文abc", "abc中文", "abc中文def", " 中文", "  中文", "\t中文", ".中文", "a,中文", ",.中文", "中文.", "中文 abc",
    "カーテン", "ひらがなカタカナ漢字", "한국어 text", "々々", "〆切", "ㄅㄆ中", "中ㄅ", "ｱｲｳ", "ﾟ中",
    "x 中 y", "中1234中", "1中2", "中's", "it's中", "中'S", "don't", "DON'T", "'s", " 's", "x's's",
    "naïve中", "Ωmega中文", "中\n文", "中\r\n\r\n  文", "中  \n文", "\n\n中", "中;\n\n", "12345678",
    "  foo", "a.foo", " .foo", "Hello World", "x　y", "中　文", "𠀀𠀁a", "a𠀀", "中́文",
]


def main(out):
    rx = regex.compile(DEEPSEEK_RE)
    with open(out, "w") as f:
        f.write("# DeepSeek-style splits from regex %s; each line: [text, [fragments]]\n" % regex.__version__)
        for s in EXAMPLES:
            f.write(json.dumps([s, rx.findall(s)], ensure_ascii=False) + "\n")
    print(len(EXAMPLES), "pins ->", out)


if __name__ == "__main__":
    main(os.path.join(os.path.dirname(os.path.abspath(__file__)), "pretoken_pins_deepseek.txt"))
